// kda_tc_prefill.cu -- chunked KDA prefill on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM), bf16 inputs, dk = dv = 128, chunk 64.
//
// Chunked form of the recurrence (delta rule with a diagonal gate, "From KV
// Cache to Depth Attention", Technical Details; FlashKDA's unrolling in
// chunks, "Kimi K3: The Manos, The Mythos, The Legendos", bullet list).  For
// a chunk of L <= 64 tokens with start state S0, G_i = sum_{m<=i} log alpha_m
// per key channel and Gamma = exp(G):
//
//   Kp = K^ o Gamma,  Kn = K^ o Gamma^{-1},  Qp = Q^ o Gamma,  Kr = K^ o Gamma_L/Gamma
//   [A_kk ; A_qk] = [Kp ; Qp] Kn^T            (tensor cores, M=128 N=64 K=128)
//   A_kk <- diag(beta) strict-lower(A_kk),   A_qk <- lower(A_qk)
//   Tb = (I + A_kk)^{-1} diag(beta)           (CUDA cores, blocked substitution)
//   [W | U~] = Tb [Kp | V]                    (tensor cores, M=64 N=256 K=64)
//   per chunk, in order:  U = U~ - W S0
//                         O = scale (Qp S0 + A_qk U)
//                         S_end = Diag(Gamma_L) S0 + Kr^T U
//
// K2 (tc_intra): one CTA per (chunk, head), fully parallel.  It reads the raw
//   q, k, g, v, b tiles, forms the operands above and writes one record per
//   (chunk, head) whose tiles are already in the shared-memory operand layout
//   of K3, so K3 moves them with single bulk (TMA engine) copies.
// K3 (tc_inter): one CTA per (sequence, head, 32-column slice of S), walking
//   the chunks in order with S in TMEM (fp32 accumulator) and a bf16 copy of
//   S in shared memory as the MMA operand; records are prefetched two
//   chunks ahead by bulk copies.  U enters its MMAs as a bf16 hi + lo pair,
//   so the value path keeps ~16 mantissa bits.
//
// The factored exponentials exp(G_i) exp(-G_j) stay finite while a chunk's
// total log-decay per channel is above about -80 (alpha products down to
// ~1e-35 over 64 tokens); the fp32 CUDA-core path has no such limit.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

// ---------------------------------------------------------------- record layout
// Per (chunk, head), bytes:
//   AW  [128][128] bf16, K-major R=128: rows 0-63 W, rows 64-127 Qp
//   AK  [128][64]  bf16, K-major R=128: Kr^T (row = key channel, K = token)
//   AQ  [64][64]   bf16, K-major R=64:  A_qk (row i, K = j)
//   UT  fp32, element (i, e) at ((e/4)*64 + i)*4 + e%4   (U~)
//   GL  [128] fp32: Gamma_L
struct Rec {
  static constexpr uint32_t AW = 0;
  static constexpr uint32_t AK = AW + 128 * 128 * 2;
  static constexpr uint32_t AQ = AK + 128 * 64 * 2;
  static constexpr uint32_t UT = AQ + 64 * 64 * 2;
  static constexpr uint32_t GL = UT + 64 * 128 * 4;
  static constexpr uint32_t BYTES = GL + 128 * 4;
};
static_assert(Rec::BYTES % 256 == 0, "records stay 256-byte aligned");

constexpr int kThreads = 128;
constexpr uint32_t kD = 128;  // dk = dv

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void st_smem16(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

__device__ __forceinline__ void flag(int32_t* status, int32_t f) { atomicOr(status, f); }

// ================================================================ K2: intra-chunk
// shared memory of tc_intra (bytes)
struct K2Smem {
  static constexpr uint32_t A1 = 0;                    // [Kp;Qp] -> [W;Qp], R=128, K=128
  static constexpr uint32_t B1 = A1 + 128 * 128 * 2;   // Kn, R=64, K=128
  static constexpr uint32_t B2 = B1 + 64 * 128 * 2;    // [Kp^T; V^T], R=256, K=64
  static constexpr uint32_t A2 = B2 + 256 * 64 * 2;    // Tb, R=64, K=64
  static constexpr uint32_t AKK = A2 + 64 * 64 * 2;    // fp32 [64][68] (A_kk)
  static constexpr uint32_t X = AKK + 64 * 68 * 4;     // fp32 [3][16][16] block-product scratch
  static constexpr uint32_t MISC = X + 3 * 256 * 4;    // inv_q, inv_k, beta [64] + partial [2][4][64]
  static constexpr uint32_t BYTES = MISC + (3 * 64 + 2 * 4 * 64) * 4;
  // T = (I + A_kk)^{-1} (fp32 [64][64]) reuses B1 once the first MMA has read Kn
};
constexpr int kAs = 68;  // row stride of A_kk
constexpr int kTs = 64;  // row stride of T

// Inverse of the unit lower-triangular 64x64 matrix (I + A) (A strictly
// lower, fp32 in shared memory, row stride kAs), blocked in 16x16 tiles:
// diagonal tiles by forward substitution, then T_ij = -T_ii sum_k A_ik T_kj
// for the off-diagonal tiles by block distance.  Result in T (stride kTs).
__device__ void tri_inverse_64(const float* __restrict__ A, float* __restrict__ T, float* X) {
  const int tid = threadIdx.x;
  // diagonal tiles: thread (d, jj) owns column jj of tile d
  if (tid < 64) {
    const int d = tid >> 4, jj = tid & 15, j = 16 * d + jj;
    float col[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      float acc = (ii == jj) ? 1.f : 0.f;
      if (ii > jj) {
#pragma unroll
        for (int m = 0; m < 16; ++m)
          if (m < ii) acc -= A[(16 * d + ii) * kAs + 16 * d + m] * col[m];
      }
      col[ii] = acc;
    }
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) T[(16 * d + ii) * kTs + j] = col[ii];
  }
  // zero the strictly upper off-diagonal tiles
  for (int idx = tid; idx < 64 * 64; idx += kThreads) {
    const int r = idx >> 6, c = idx & 63;
    if ((c >> 4) > (r >> 4)) T[r * kTs + c] = 0.f;
  }
  __syncthreads();
  for (int dist = 1; dist < 4; ++dist) {
    const int ntiles = 4 - dist;  // tiles (i, j = i - dist), i = dist..3
    // X_ij = sum_{k=j}^{i-1} A_ik T_kj  (16x16 each), into X [ntiles][16][16]
    for (int idx = tid; idx < ntiles * 256; idx += kThreads) {
      const int t = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      const int bi = dist + t, bj = t;
      const int row = 16 * bi + r, colg = 16 * bj + c;
      float acc = 0.f;
      for (int kk = 16 * bj; kk < 16 * bi; ++kk) acc += A[row * kAs + kk] * T[kk * kTs + colg];
      X[idx] = acc;
    }
    __syncthreads();
    // T_ij = -T_ii X_ij
    for (int idx = tid; idx < ntiles * 256; idx += kThreads) {
      const int t = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      const int bi = dist + t, bj = t;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc += T[(16 * bi + r) * kTs + 16 * bi + m] * X[(t << 8) + (m << 4) + c];
      T[(16 * bi + r) * kTs + 16 * bj + c] = -acc;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_intra(ChunkParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base;

  const int64_t cidx = blockIdx.x;
  if (cidx >= p.meta->total_chunks) return;
  const int h = blockIdx.y, H = p.H;
  const Chunk ch = p.chunks[cidx];
  const int len = ch.len;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tb = lane >> 2;                 // token block: tokens 8tb .. 8tb+7
  const int cb = warp * 4 + (lane & 3);     // channel block: channels 8cb .. 8cb+7
  const int i0 = 8 * tb, c0 = 8 * cb;

  uint8_t* A1 = sm + K2Smem::A1;
  uint8_t* B1 = sm + K2Smem::B1;
  uint8_t* B2 = sm + K2Smem::B2;
  uint8_t* A2 = sm + K2Smem::A2;
  float* AKK = reinterpret_cast<float*>(sm + K2Smem::AKK);
  float* TT = reinterpret_cast<float*>(sm + K2Smem::B1);
  float* XS = reinterpret_cast<float*>(sm + K2Smem::X);
  float* inv_q = reinterpret_cast<float*>(sm + K2Smem::MISC);
  float* inv_k = inv_q + 64;
  float* beta = inv_k + 64;
  float* part = beta + 64;  // [2][4][64]

  uint8_t* rec = reinterpret_cast<uint8_t*>(p.inter) + ((size_t)cidx * H + h) * Rec::BYTES;

  if (warp == 0) tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    mbar_init_fence();
  }

  const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
  const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(p.g);
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(p.b);
  auto row_ptr = [&](const __nv_bfloat16* base, int i) {
    return reinterpret_cast<const uint4*>(base + ((ch.tok0 + i) * H + h) * (int64_t)kD + c0);
  };

  // ---- 1. log-decay running sums G (8 tokens x 8 channels per thread)
  float G[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = i0 + r;
    const uint4 gr = i < len ? __ldg(row_ptr(gg, i)) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float la0 = i < len ? log_alpha_of(bf16_lo(w[j])) : 0.f;
      const float la1 = i < len ? log_alpha_of(bf16_hi(w[j])) : 0.f;
      G[r][2 * j] = (r ? G[r - 1][2 * j] : 0.f) + la0;
      G[r][2 * j + 1] = (r ? G[r - 1][2 * j + 1] : 0.f) + la1;
    }
  }
  // exclusive scan of the block totals over the 8 token blocks (lanes 4 apart)
  float GL[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float tot = G[7][j];
    float inc = tot;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += y;
    }
    const float ex = inc - tot;
#pragma unroll
    for (int r = 0; r < 8; ++r) G[r][j] += ex;
    GL[j] = __shfl_sync(0xffffffffu, inc, 28 + (lane & 3));
  }

  // ---- 2. L2 norms of q and k per token (8 channels here, 4 lanes, 4 warps)
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = i0 + r;
    const uint4 qr = i < len ? __ldg(row_ptr(gq, i)) : make_uint4(0, 0, 0, 0);
    const uint4 kr = i < len ? __ldg(row_ptr(gk, i)) : make_uint4(0, 0, 0, 0);
    float sq = 0.f, sk = 0.f;
    const uint32_t wq[4] = {qr.x, qr.y, qr.z, qr.w};
    const uint32_t wk[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sq += bf16_lo(wq[j]) * bf16_lo(wq[j]) + bf16_hi(wq[j]) * bf16_hi(wq[j]);
      sk += bf16_lo(wk[j]) * bf16_lo(wk[j]) + bf16_hi(wk[j]) * bf16_hi(wk[j]);
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
    if ((lane & 3) == 0) {
      part[warp * 64 + i0 + r] = sq;
      part[256 + warp * 64 + i0 + r] = sk;
    }
  }
  __syncthreads();
  if (tid < 64) {
    const int i = tid;
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      sq += part[w * 64 + i];
      sk += part[256 + w * 64 + i];
    }
    inv_q[i] = inv_norm_of(sq);
    inv_k[i] = inv_norm_of(sk);
    beta[i] = i < len ? beta_of(__bfloat162float(gb[(ch.tok0 + i) * H + h])) : 0.f;
  }
  __syncthreads();

  // ---- 3. operands: Kp, Qp (A1), Kn (B1), Kp^T (B2 rows 0-127), Kr^T (record AK)
  {
    uint32_t kpT[8][4], krT[8][4];  // transposed 8x8 blocks, bf16 pairs (token r, r+1)
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r;
      const uint4 qr = i < len ? __ldg(row_ptr(gq, i)) : make_uint4(0, 0, 0, 0);
      const uint4 kr = i < len ? __ldg(row_ptr(gk, i)) : make_uint4(0, 0, 0, 0);
      const float ik = inv_k[i], iq = inv_q[i];
      const uint32_t wq[4] = {qr.x, qr.y, qr.z, qr.w};
      const uint32_t wk[4] = {kr.x, kr.y, kr.z, kr.w};
      float kp[8], qp[8], kn[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float kh = (j & 1 ? bf16_hi(wk[j >> 1]) : bf16_lo(wk[j >> 1])) * ik;
        const float qh = (j & 1 ? bf16_hi(wq[j >> 1]) : bf16_lo(wq[j >> 1])) * iq;
        const float eg = expf(G[r][j]);
        kp[j] = kh * eg;
        qp[j] = qh * eg;
        kn[j] = kh * expf(-G[r][j]);
        const float krv = kh * expf(GL[j] - G[r][j]);
        const uint32_t bp = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(kp[j]));
        const uint32_t br = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(krv));
        if (r & 1) {
          kpT[j][r >> 1] |= bp << 16;
          krT[j][r >> 1] |= br << 16;
        } else {
          kpT[j][r >> 1] = bp;
          krT[j][r >> 1] = br;
        }
      }
      st_smem16(A1, kmajor_off(i, c0, 128),
                make_uint4(pack_bf16(kp[0], kp[1]), pack_bf16(kp[2], kp[3]),
                           pack_bf16(kp[4], kp[5]), pack_bf16(kp[6], kp[7])));
      st_smem16(A1, kmajor_off(64 + i, c0, 128),
                make_uint4(pack_bf16(qp[0], qp[1]), pack_bf16(qp[2], qp[3]),
                           pack_bf16(qp[4], qp[5]), pack_bf16(qp[6], qp[7])));
      st_smem16(B1, kmajor_off(i, c0, 64),
                make_uint4(pack_bf16(kn[0], kn[1]), pack_bf16(kn[2], kn[3]),
                           pack_bf16(kn[4], kn[5]), pack_bf16(kn[6], kn[7])));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      st_smem16(B2, kmajor_off(c0 + j, i0, 256), make_uint4(kpT[j][0], kpT[j][1], kpT[j][2], kpT[j][3]));
      *reinterpret_cast<uint4*>(rec + Rec::AK + kmajor_off(c0 + j, i0, 128)) =
          make_uint4(krT[j][0], krT[j][1], krT[j][2], krT[j][3]);
    }
  }
  // ---- 4. V^T into B2 rows 128-255 (exact bf16, transposed in registers)
  {
    uint16_t vv[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = i0 + r;
      uint4 x = i < len ? __ldg(row_ptr(gv, i)) : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        vv[r][2 * j] = (uint16_t)(w[j] & 0xffffu);
        vv[r][2 * j + 1] = (uint16_t)(w[j] >> 16);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int r2 = 0; r2 < 4; ++r2) w[r2] = (uint32_t)vv[2 * r2][j] | ((uint32_t)vv[2 * r2 + 1][j] << 16);
      st_smem16(B2, kmajor_off(128 + c0 + j, i0, 256), make_uint4(w[0], w[1], w[2], w[3]));
    }
  }
  // Gamma_L to the record (token block 7 holds the chunk total)
  if (tb == 7) {
    float* gl = reinterpret_cast<float*>(rec + Rec::GL) + c0;
    *reinterpret_cast<float4*>(gl) = make_float4(expf(GL[0]), expf(GL[1]), expf(GL[2]), expf(GL[3]));
    *reinterpret_cast<float4*>(gl + 4) = make_float4(expf(GL[4]), expf(GL[5]), expf(GL[6]), expf(GL[7]));
  }

  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  bool ok = true;

  // ---- 5. [A_kk ; A_qk] = [Kp ; Qp] Kn^T   (M=128, N=64, K=128)
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma_bf16(tmem, sdesc(smem_u32(A1) + s * 2 * 128 * 16, 128 * 16, 128),
               sdesc(smem_u32(B1) + s * 2 * 64 * 16, 64 * 16, 128), id, s > 0);
    mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(mbar_wait(&bar_mma, 0, kWaitLimitNs));
  fence_after_sync();
  if (ok) {
    float d[64];
#pragma unroll
    for (int c = 0; c < 64; c += 16) tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c, d + c);
    tmem_ld_wait();
    if (warp < 2) {
      const int i = 32 * warp + lane;
      const float bi = beta[i];
#pragma unroll
      for (int j = 0; j < 64; j += 4)
        *reinterpret_cast<float4*>(AKK + i * kAs + j) =
            make_float4(j + 0 < i ? bi * d[j] : 0.f, j + 1 < i ? bi * d[j + 1] : 0.f,
                        j + 2 < i ? bi * d[j + 2] : 0.f, j + 3 < i ? bi * d[j + 3] : 0.f);
    } else {
      const int i = 32 * (warp - 2) + lane;
      const bool live = i < len;
#pragma unroll
      for (int jb = 0; jb < 8; ++jb) {
        float a[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) a[t] = (live && 8 * jb + t <= i) ? d[8 * jb + t] : 0.f;
        *reinterpret_cast<uint4*>(rec + Rec::AQ + kmajor_off(i, 8 * jb, 64)) =
            make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                       pack_bf16(a[6], a[7]));
      }
    }
  }
  fence_before_sync();
  __syncthreads();

  // ---- 6. Tb = (I + A_kk)^{-1} diag(beta) -> A2 (bf16, K-major R=64)
  if (ok) {
    tri_inverse_64(AKK, TT, XS);
    for (int idx = tid; idx < 64 * 8; idx += kThreads) {
      const int i = idx >> 3, jb = idx & 7;
      const float* t = TT + i * kTs + 8 * jb;
      const float* bb = beta + 8 * jb;
      st_smem16(A2, kmajor_off(i, 8 * jb, 64),
                make_uint4(pack_bf16(t[0] * bb[0], t[1] * bb[1]), pack_bf16(t[2] * bb[2], t[3] * bb[3]),
                           pack_bf16(t[4] * bb[4], t[5] * bb[5]), pack_bf16(t[6] * bb[6], t[7] * bb[7])));
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- 7. [W | U~] = Tb [Kp | V]   (M=64, N=256, K=64)
  if (ok && tid == 0) {
    const uint32_t id = idesc_bf16(64, 256);
#pragma unroll
    for (int s = 0; s < 4; ++s)
      mma_bf16(tmem, sdesc(smem_u32(A2) + s * 2 * 64 * 16, 64 * 16, 128),
               sdesc(smem_u32(B2) + s * 2 * 256 * 16, 256 * 16, 128), id, s > 0);
    mma_commit(&bar_mma);
  }
  ok = __syncthreads_and(ok && mbar_wait(&bar_mma, 1, kWaitLimitNs));
  fence_after_sync();
  if (ok) {
    // M=64 accumulator: row r sits in TMEM lane (r/16)*32 + r%16
    const int i = 16 * warp + (lane & 15);
    const bool row_lane = lane < 16;
    const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
    for (int c = 0; c < 128; c += 16) {
      float d[16];
      tmem_ld16(ta + c, d);
      tmem_ld_wait();
      if (row_lane) {
        st_smem16(A1, kmajor_off(i, c, 128),
                  make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                             pack_bf16(d[6], d[7])));
        st_smem16(A1, kmajor_off(i, c + 8, 128),
                  make_uint4(pack_bf16(d[8], d[9]), pack_bf16(d[10], d[11]),
                             pack_bf16(d[12], d[13]), pack_bf16(d[14], d[15])));
      }
    }
#pragma unroll
    for (int c = 0; c < 128; c += 16) {
      float d[16];
      tmem_ld16(ta + 128 + c, d);
      tmem_ld_wait();
      if (row_lane) {
        float* ut = reinterpret_cast<float*>(rec + Rec::UT);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<float4*>(ut + (((c >> 2) + q4) * 64 + i) * 4) =
              make_float4(d[4 * q4], d[4 * q4 + 1], d[4 * q4 + 2], d[4 * q4 + 3]);
      }
    }
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    if (ok) {
      bulk_s2g(rec + Rec::AW, A1, 128 * 128 * 2);
      bulk_commit();
      bulk_wait_all();
    } else {
      flag(p.status, kFlagTimeout);
    }
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ================================================================ K3: inter-chunk
constexpr int kNs = 32;  // state columns per CTA

struct K3Smem {
  // one ring slot: AW (32 KB) | AK (16 KB) | AQ128 (16 KB, rows 64-127 used) | UT slice | GL
  static constexpr uint32_t AW = 0;
  static constexpr uint32_t AK = AW + 128 * 128 * 2;
  static constexpr uint32_t AQ = AK + 128 * 64 * 2;
  static constexpr uint32_t UT = AQ + 128 * 64 * 2;
  static constexpr uint32_t GL = UT + 64 * kNs * 4;
  static constexpr uint32_t SLOT = GL + 128 * 4;
  static constexpr uint32_t SOP = 2 * SLOT;                 // S^T operand, R=kNs, K=128
  static constexpr uint32_t UHI = SOP + kNs * 128 * 2;       // U operand, R=kNs, K=64
  static constexpr uint32_t ULO = UHI + kNs * 64 * 2;
  static constexpr uint32_t BYTES = ULO + kNs * 64 * 2;
  static constexpr uint32_t TX = 128 * 128 * 2 + 128 * 64 * 2 + 64 * 64 * 2 + 64 * kNs * 4 + 128 * 4;
};

__device__ __forceinline__ void k3_issue_loads(const ChunkParams& p, uint8_t* slot, uint64_t* bar,
                                               int64_t cidx, int h, int n0) {
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, K3Smem::TX);
  bulk_g2s(slot + K3Smem::AW, rec + Rec::AW, 128 * 128 * 2, bar);
  bulk_g2s(slot + K3Smem::AK, rec + Rec::AK, 128 * 64 * 2, bar);
  // A_qk rows into rows 64-127 of a R=128 K-major tile: the second 1 KB of each 2 KB K-block
#pragma unroll
  for (int kb = 0; kb < 8; ++kb)
    bulk_g2s(slot + K3Smem::AQ + kb * 2048 + 1024, rec + Rec::AQ + kb * 1024, 1024, bar);
  bulk_g2s(slot + K3Smem::UT, rec + Rec::UT + (n0 / 4) * 64 * 16, 64 * kNs * 4, bar);
  bulk_g2s(slot + K3Smem::GL, rec + Rec::GL, 128 * 4, bar);
}

__global__ void __launch_bounds__(kThreads, 1)
tc_inter(ChunkParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar_full[2];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base;

  const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * kNs;
  const int H = p.H, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c_begin = p.seq_chunk_begin[s], c_end = p.seq_chunk_begin[s + 1];
  if (c_end > c_begin && p.meta->total_chunks == 0) return;  // chunk table overflowed
  const int64_t nchunks = c_end - c_begin;

  uint8_t* SOP = sm + K3Smem::SOP;
  uint8_t* UHI = sm + K3Smem::UHI;
  uint8_t* ULO = sm + K3Smem::ULO;

  // zero both ring slots once: rows 0-63 of the AQ tiles are never loaded
  for (uint32_t off = tid * 16; off < 2 * K3Smem::SLOT; off += kThreads * 16)
    *reinterpret_cast<uint4*>(sm + off) = make_uint4(0, 0, 0, 0);
  if (warp == 0) tmem_alloc(&tmem_base, 2 * kNs);
  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_mma, 1);
    mbar_init_fence();
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t D1 = tmem;          // [W;Qp] S0, then + A_qk U in lanes 64-127
  const uint32_t DS = tmem + kNs;    // the state slice, lane = key channel
  const uint32_t lane_off = (uint32_t)(32 * warp) << 16;

  if (tid == 0) {
    for (int64_t it = 0; it < 2 && it < nchunks; ++it)
      k3_issue_loads(p, sm + it * K3Smem::SLOT, &bar_full[it], c_begin + it, h, n0);
  }

  // initial state slice: TMEM (fp32) and the bf16 operand copy
  const int c = tid;  // key channel == TMEM lane
  const size_t sbase = ((size_t)s * H + h) * kD * kD;
  {
    float v[kNs];
#pragma unroll
    for (int n = 0; n < kNs; n += 4) {
      float4 x = p.initial_state
                     ? *reinterpret_cast<const float4*>(p.initial_state + sbase + (size_t)c * kD + n0 + n)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      v[n] = x.x; v[n + 1] = x.y; v[n + 2] = x.z; v[n + 3] = x.w;
    }
    tmem_st16(DS + lane_off, v);
    tmem_st16(DS + lane_off + 16, v + 16);
    tmem_st_wait();
#pragma unroll
    for (int n = 0; n < kNs; ++n)
      *reinterpret_cast<__nv_bfloat16*>(SOP + kmajor_off(n, c, kNs)) = __float2bfloat16_rn(v[n]);
  }

  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
  const float scale = p.scale;
  uint32_t mma_phase = 0;
  bool ok = true;
  for (int64_t it = 0; it < nchunks && ok; ++it) {
    const int slot_i = (int)(it & 1);
    uint8_t* slot = sm + slot_i * K3Smem::SLOT;
    const Chunk ch = p.chunks[c_begin + it];
    // S operand (previous iteration) and this slot are ready
    fence_async_smem();
    fence_before_sync();
    ok = __syncthreads_and(mbar_wait(&bar_full[slot_i], (uint32_t)((it >> 1) & 1), kWaitLimitNs));
    fence_after_sync();
    if (!ok) break;
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, kNs);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(D1, sdesc(smem_u32(slot + K3Smem::AW) + k * 2 * 128 * 16, 128 * 16, 128),
                 sdesc(smem_u32(SOP) + k * 2 * kNs * 16, kNs * 16, 128), id, k > 0);
      mma_commit(&bar_mma);
    }
    // retention of the carried state while MMA1 runs: S <- Diag(Gamma_L) S
    {
      const float gl = reinterpret_cast<const float*>(slot + K3Smem::GL)[c];
      float v[kNs];
      tmem_ld16(DS + lane_off, v);
      tmem_ld16(DS + lane_off + 16, v + 16);
      tmem_ld_wait();
#pragma unroll
      for (int n = 0; n < kNs; ++n) v[n] *= gl;
      tmem_st16(DS + lane_off, v);
      tmem_st16(DS + lane_off + 16, v + 16);
      tmem_st_wait();
    }
    fence_before_sync();
    ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase, kWaitLimitNs));
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    if (warp < 2) {
      // U = U~ - W S0 for token i = lane row, split into bf16 hi + lo
      const int i = tid;
      float d[kNs];
      tmem_ld16(D1 + lane_off, d);
      tmem_ld16(D1 + lane_off + 16, d + 16);
      tmem_ld_wait();
      const float* ut = reinterpret_cast<const float*>(slot + K3Smem::UT);
#pragma unroll
      for (int q4 = 0; q4 < kNs / 4; ++q4) {
        const float4 u4 = *reinterpret_cast<const float4*>(ut + (q4 * 64 + i) * 4);
        const float uu[4] = {u4.x - d[4 * q4], u4.y - d[4 * q4 + 1], u4.z - d[4 * q4 + 2],
                             u4.w - d[4 * q4 + 3]};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int n = 4 * q4 + t;
          const __nv_bfloat16 hi = __float2bfloat16_rn(uu[t]);
          const __nv_bfloat16 lo = __float2bfloat16_rn(uu[t] - __bfloat162float(hi));
          *reinterpret_cast<__nv_bfloat16*>(UHI + kmajor_off(n, i, kNs)) = hi;
          *reinterpret_cast<__nv_bfloat16*>(ULO + kmajor_off(n, i, kNs)) = lo;
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, kNs);
      // S += Kr^T U   and   D1[64..127] += A_qk U   (U as hi + lo)
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t ub = smem_u32(part ? ULO : UHI);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t bdesc = sdesc(ub + k * 2 * kNs * 16, kNs * 16, 128);
          mma_bf16(DS, sdesc(smem_u32(slot + K3Smem::AK) + k * 2 * 128 * 16, 128 * 16, 128), bdesc,
                   id, 1);
          mma_bf16(D1, sdesc(smem_u32(slot + K3Smem::AQ) + k * 2 * 128 * 16, 128 * 16, 128), bdesc,
                   id, 1);
        }
      }
      mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase, kWaitLimitNs));
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    // this slot is free: prefetch chunk it + 2 into it
    if (tid == 0 && it + 2 < nchunks)
      k3_issue_loads(p, slot, &bar_full[slot_i], c_begin + it + 2, h, n0);
    // outputs: o = scale * (Qp S0 + A_qk U) from lanes 64-127
    if (warp >= 2) {
      const int i = tid - 64;
      float d[kNs];
      tmem_ld16(D1 + lane_off, d);
      tmem_ld16(D1 + lane_off + 16, d + 16);
      tmem_ld_wait();
      if (i < ch.len) {
        uint4* dst = reinterpret_cast<uint4*>(o + ((ch.tok0 + i) * H + h) * (int64_t)kD + n0);
#pragma unroll
        for (int q8 = 0; q8 < kNs / 8; ++q8)
          dst[q8] = make_uint4(pack_bf16(scale * d[8 * q8], scale * d[8 * q8 + 1]),
                               pack_bf16(scale * d[8 * q8 + 2], scale * d[8 * q8 + 3]),
                               pack_bf16(scale * d[8 * q8 + 4], scale * d[8 * q8 + 5]),
                               pack_bf16(scale * d[8 * q8 + 6], scale * d[8 * q8 + 7]));
      }
    }
    // new state: bf16 operand copy, snapshot if this chunk ends at one
    {
      float v[kNs];
      tmem_ld16(DS + lane_off, v);
      tmem_ld16(DS + lane_off + 16, v + 16);
      tmem_ld_wait();
#pragma unroll
      for (int n = 0; n < kNs; ++n)
        *reinterpret_cast<__nv_bfloat16*>(SOP + kmajor_off(n, c, kNs)) = __float2bfloat16_rn(v[n]);
      if (ch.snap_slot >= 0 && p.snapshots) {
        float* dst = p.snapshots + ((size_t)ch.snap_slot * H + h) * kD * kD + (size_t)c * kD + n0;
#pragma unroll
        for (int n = 0; n < kNs; n += 4)
          *reinterpret_cast<float4*>(dst + n) = make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
      }
    }
  }
  if (!ok && tid == 0) flag(p.status, kFlagTimeout);
  if (p.final_state && ok) {
    float v[kNs];
    tmem_ld16(DS + lane_off, v);
    tmem_ld16(DS + lane_off + 16, v + 16);
    tmem_ld_wait();
    float* dst = p.final_state + sbase + (size_t)c * kD + n0;
#pragma unroll
    for (int n = 0; n < kNs; n += 4)
      *reinterpret_cast<float4*>(dst + n) = make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * kNs);
}

}  // namespace

const bool kHaveTensorCorePath = true;

size_t tc_record_bytes() { return Rec::BYTES; }

cudaError_t launch_tc_prefill(const ChunkParams& p, cudaStream_t stream, cudaEvent_t mid) {
  cudaError_t e = cudaFuncSetAttribute(tc_intra, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)K2Smem::BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_inter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)K3Smem::BYTES);
  if (e != cudaSuccess) return e;
  if (p.max_chunks > 0) {
    dim3 grid((unsigned)p.max_chunks, (unsigned)p.H);
    tc_intra<<<grid, kThreads, K2Smem::BYTES, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (mid) {
    e = cudaEventRecord(mid, stream);
    if (e != cudaSuccess) return e;
  }
  dim3 grid2((unsigned)p.num_seqs, (unsigned)p.H, (unsigned)(kD / kNs));
  tc_inter<<<grid2, kThreads, K3Smem::BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
