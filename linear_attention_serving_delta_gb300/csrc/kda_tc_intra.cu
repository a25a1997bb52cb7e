// kda_tc_intra.cu -- K2, the intra-chunk kernel of the tensor-core prefill.
//
// Persistent, two CTAs of 256 threads per SM.  For each (chunk, head) item
// every thread owns 4 consecutive tokens x 8 channels: its q, k, g, v rows
// (16-byte loads, prefetched during the previous item), the cumulative decay
// Gamma as a product scan (in registers, then across the 16 token blocks with
// shuffles), normalised q and k, and the operands written with 16-byte
// shared stores straight into the tcgen05 layouts (K-major where a row of 8
// channels is one core-matrix row, MN-major where 8 channels of one token
// are).  Then:
//   MMA 1 (M=128, N=64, K=128):  [A_kk ; A_qk] = [Kp ; Qp] Kn^T  -> TMEM
//   CUDA cores: T = (I + A_kk)^{-1}, two-level blocked inverse
//   MMA 2 (M=64, N=256, K=64):   [W | U~] = T diag(beta) [Kp | V] -> TMEM
// and the record of kda_tc_common.cuh is written (AW with one bulk copy).
// The math is stated in kda_tc_common.cuh.
#include "kda_tc_common.cuh"

namespace kda {
namespace tcp {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kAs = 68;  // row stride (floats) of A_kk in shared memory
constexpr int kTs = 64;  // row stride (floats) of T
constexpr uint32_t kB2Sbo = 8 * 128;  // B2 MN-major: 8 K-groups (64 tokens) per MN-group

struct Smem {
  static constexpr uint32_t A1 = 0;                    // [Kp;Qp] -> [W;Qp], R=128, K=128
  static constexpr uint32_t B1 = A1 + 128 * 128 * 2;   // Kn, R=64, K=128; then T fp32 [64][64]
  static constexpr uint32_t B2 = B1 + 64 * 128 * 2;    // [Kp | V] as MN-major (n, token), N=256
  static constexpr uint32_t A2 = B2 + 256 * 64 * 2;    // inverse scratch; then Tb, R=64, K=64
  static constexpr uint32_t AKK = A2 + 64 * 64 * 2;    // fp32 [64][kAs]
  static constexpr uint32_t MISC = AKK + 64 * kAs * 4; // inv_q, inv_k, beta [64]; part [2][8][64]
  static constexpr uint32_t BYTES = MISC + (3 * 64 + 2 * 8 * 64) * 4;
};

__device__ __forceinline__ void st_s16(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}

// T = (I + A)^{-1} for strictly lower-triangular A (64x64, stride kAs).
// Level 0: the four 16x16 diagonal tiles by forward substitution (a thread
// per column).  Level 1: the two 16x16 tiles below them inside each 32x32
// half, T10 = -T11 A10 T00.  Level 2: the lower-left 32x32 tile,
// T = -T_hi A T_lo.  X: scratch of 32x32 floats.  256 threads.
__device__ void tri_inverse_64(const float* __restrict__ A, float* __restrict__ T,
                               float* __restrict__ X) {
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int d = tid >> 4, jj = tid & 15, j = 16 * d + jj;
    float col[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) col[m] = 0.f;
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      const float4* ar = reinterpret_cast<const float4*>(A + (16 * d + ii) * kAs + 16 * d);
      float acc[4] = {ii == jj ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 a = ar[q4];
        acc[0] -= a.x * col[4 * q4];
        acc[1] -= a.y * col[4 * q4 + 1];
        acc[2] -= a.z * col[4 * q4 + 2];
        acc[3] -= a.w * col[4 * q4 + 3];
      }
      col[ii] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) T[(16 * d + ii) * kTs + j] = col[ii];
  } else {
    // tiles strictly above the diagonal are zero
    for (int idx = tid - 64; idx < 6 * 256; idx += kThreads - 64) {
      const int t = idx >> 8, e = idx & 255;
      const int bi = t < 3 ? 0 : (t < 5 ? 1 : 2);
      const int bj = t < 3 ? t + 1 : (t < 5 ? t - 1 : 3);
      T[(16 * bi + (e >> 4)) * kTs + 16 * bj + (e & 15)] = 0.f;
    }
  }
  __syncthreads();
  // level 1: P = 0, 1 -> tile rows 32P+16.., cols 32P..
  {
    const int P = tid >> 7, rr = (tid >> 3) & 15, cc = (tid & 7) * 2;
    const int r0 = 32 * P + 16, c0 = 32 * P;
    float x0 = 0.f, x1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float a = A[(r0 + rr) * kAs + c0 + m];
      const float2 t = *reinterpret_cast<const float2*>(T + (c0 + m) * kTs + c0 + cc);
      x0 += a * t.x;
      x1 += a * t.y;
    }
    X[P * 256 + rr * 16 + cc] = x0;
    X[P * 256 + rr * 16 + cc + 1] = x1;
    __syncthreads();
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const float t = T[(r0 + rr) * kTs + r0 + m];
      y0 += t * X[P * 256 + m * 16 + cc];
      y1 += t * X[P * 256 + m * 16 + cc + 1];
    }
    T[(r0 + rr) * kTs + c0 + cc] = -y0;
    T[(r0 + rr) * kTs + c0 + cc + 1] = -y1;
  }
  __syncthreads();
  // level 2: rows 32..63, cols 0..31, 2x2 outputs per thread
  {
    const int rr = (tid >> 4) * 2, cc = (tid & 15) * 2;
    float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float a0 = A[(32 + rr) * kAs + m], a1 = A[(33 + rr) * kAs + m];
      const float2 t = *reinterpret_cast<const float2*>(T + m * kTs + cc);
      x00 += a0 * t.x; x01 += a0 * t.y;
      x10 += a1 * t.x; x11 += a1 * t.y;
    }
    X[rr * 32 + cc] = x00; X[rr * 32 + cc + 1] = x01;
    X[(rr + 1) * 32 + cc] = x10; X[(rr + 1) * 32 + cc + 1] = x11;
    __syncthreads();
    float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
#pragma unroll 8
    for (int m = 0; m < 32; ++m) {
      const float t0 = T[(32 + rr) * kTs + 32 + m], t1 = T[(33 + rr) * kTs + 32 + m];
      const float2 x = *reinterpret_cast<const float2*>(X + m * 32 + cc);
      y00 += t0 * x.x; y01 += t0 * x.y;
      y10 += t1 * x.x; y11 += t1 * x.y;
    }
    T[(32 + rr) * kTs + cc] = -y00; T[(32 + rr) * kTs + cc + 1] = -y01;
    T[(33 + rr) * kTs + cc] = -y10; T[(33 + rr) * kTs + cc + 1] = -y11;
  }
  __syncthreads();
}

// Raw rows of one work item (chunk, head) for this thread: 4 tokens (4 tb + r)
// x 8 channels of q, k, g, v, and the update logit of token `tid` (tid < 64).
struct RawRows {
  uint4 g[4], q[4], k[4], v[4];
  float b;
};

// 16-byte read-only global load kept at its place in the program (volatile),
// so a prefetch is issued where it is written and not sunk to its first use
__device__ __forceinline__ uint4 ld_nc16(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// One of the four tensors' rows (0 g, 1 q, 2 k, 3 v) of an item.  The
// prefetch of the next item is spread over the current item's phases, so
// that the load-queue back-pressure of each group drains behind compute.
__device__ __forceinline__ void load_part(const ChunkParams& p, const Chunk& ch, int h, int tb, int c0,
                                          int which, uint4* dst) {
  const void* base = which == 0 ? p.g : which == 1 ? p.q : which == 2 ? p.k : p.v;
  const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(base);
  const int H = p.H, len = ch.len;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = 4 * tb + r;
    const int64_t e = ((ch.tok0 + i) * H + h) * (int64_t)kD + c0;
    dst[r] = i < len ? ld_nc16(src + e) : make_uint4(0, 0, 0, 0);
  }
}

__device__ __forceinline__ float load_b(const ChunkParams& p, const Chunk& ch, int h, int tid) {
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(p.b);
  return (tid < 64 && tid < ch.len) ? __bfloat162float(gb[(ch.tok0 + tid) * p.H + h]) : 0.f;
}

__device__ __forceinline__ void load_rows(const ChunkParams& p, const Chunk& ch, int h, int tb, int c0,
                                          int tid, RawRows& R) {
  load_part(p, ch, h, tb, c0, 0, R.g);
  load_part(p, ch, h, tb, c0, 1, R.q);
  load_part(p, ch, h, tb, c0, 2, R.k);
  load_part(p, ch, h, tb, c0, 3, R.v);
  R.b = load_b(p, ch, h, tid);
}

// Persistent: two CTAs per SM walk the (chunk, head) items with stride
// gridDim.x.  The raw rows of the next item are loaded into the registers
// freed once the current item's operands are built, so its DRAM reads
// overlap this item's MMAs, inverse and record stores.  TMEM and the
// mbarrier are set up once per CTA.
__global__ void __launch_bounds__(kThreads, 2)
tc_intra(ChunkParams p, int64_t n_items) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_base;

  const int64_t stride = gridDim.x;
  int64_t item = blockIdx.x;
  if (item >= n_items) return;
  const int H = p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // this thread: tokens 4 tb .. 4 tb + 3, channels 8 cb .. 8 cb + 7.  Four
  // consecutive tokens per thread keep the decay scan in registers (one
  // shuffle per element); the operand stores see at most 4-way bank conflicts.
  const int tb = lane >> 1;
  const int cb = 2 * warp + (lane & 1);
  const int c0 = 8 * cb;
  const int quarter = warp & 3, half = warp >> 2;

  uint8_t* A1 = sm + Smem::A1;
  uint8_t* B1 = sm + Smem::B1;
  uint8_t* B2 = sm + Smem::B2;
  uint8_t* A2 = sm + Smem::A2;
  float* AKK = reinterpret_cast<float*>(sm + Smem::AKK);
  float* TT = reinterpret_cast<float*>(sm + Smem::B1);
  float* XS = reinterpret_cast<float*>(sm + Smem::A2);
  float* inv_q = reinterpret_cast<float*>(sm + Smem::MISC);
  float* inv_k = inv_q + 64;
  float* beta = inv_k + 64;
  float* part = beta + 64;  // [2][8][64]

  if (warp == 0) tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    mbar_init_fence();
  }

  // the pipeline: chunk entry and raw rows of the current item, chunk entry of the next
  Chunk ch = p.chunks[item / H];  // entries past the table's end have len 0
  RawRows R;
  load_rows(p, ch, (int)(item % H), tb, c0, tid, R);
  Chunk ch_next = item + stride < n_items ? p.chunks[(item + stride) / H] : Chunk{};

  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  bool ok = true;

  for (; item < n_items; item += stride) {
    const int h = (int)(item % H);
    const int64_t cidx = item / H;
    const int len = ch.len;
    if (len == 0) {  // past the end of the chunk table (uniform across the CTA)
      if (item + stride < n_items) load_rows(p, ch_next, (int)((item + stride) % H), tb, c0, tid, R);
      ch = ch_next;
      ch_next = item + 2 * stride < n_items ? p.chunks[(item + 2 * stride) / H] : Chunk{};
      continue;
    }
    uint8_t* rec = reinterpret_cast<uint8_t*>(p.inter) + ((size_t)cidx * H + h) * Rec::BYTES;

    // ---- V into B2 MN-major rows 128..255: the raw 16 bytes are one core-matrix row
#pragma unroll
    for (int r = 0; r < 4; ++r) st_s16(B2, mnmajor_off(128 + c0, 4 * tb + r, kB2Sbo), R.v[r]);

    // ---- cumulative decay Gamma_i = prod_{m<=i} alpha_m, alpha = 1 / (1 + e^g)
    // (= exp(-softplus(g))): a product over this thread's 4 tokens, then an
    // exclusive product scan across the 16 token blocks (lanes 2 apart)
    float Gm[4][8], GLm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float run = 1.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float a = 4 * tb + r < len ? alpha_fast(bf16_at(R.g[r], j)) : 1.f;
        run *= a;
        Gm[r][j] = run;
      }
      float inc = run;
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc *= y;
      }
      float ex = __shfl_up_sync(0xffffffffu, inc, 2);
      if (lane < 2) ex = 1.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) Gm[r][j] *= ex;
      GLm[j] = __shfl_sync(0xffffffffu, inc, 30 + (lane & 1));
    }

    // ---- L2 norms per token: 8 channels here, 2 per warp, 8 warps
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float xq = bf16_at(R.q[r], j), xk = bf16_at(R.k[r], j);
        sq += xq * xq;
        sk += xk * xk;
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      if ((lane & 1) == 0) {
        part[warp * 64 + 4 * tb + r] = sq;
        part[512 + warp * 64 + 4 * tb + r] = sk;
      }
    }
    if (tid < 64) beta[tid] = tid < len ? beta_of(R.b) : 0.f;
    // the previous item's record copy must have finished reading A1
    if (tid == 0) bulk_wait_read_all();
    __syncthreads();
    if (tid < 64) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        sq += part[w * 64 + tid];
        sk += part[512 + w * 64 + tid];
      }
      inv_q[tid] = inv_norm_of(sq);
      inv_k[tid] = inv_norm_of(sk);
    }
    __syncthreads();

    // ---- operands Kp, Qp (A1), Kn (B1), Kp (B2 MN-major rows 0-127), Kr (record AK, MN-major)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = 4 * tb + r;
      const float ik = inv_k[i], iq = inv_q[i];
      float kp[8], qp[8], kn[8], kx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float kh = bf16_at(R.k[r], j) * ik;
        const float qh = bf16_at(R.q[r], j) * iq;
        const float gam = Gm[r][j];
        kp[j] = kh * gam;
        qp[j] = qh * gam;
        kn[j] = __fdividef(kh, gam);
        kx[j] = kn[j] * GLm[j];
      }
      const uint4 kpv = make_uint4(pack_bf16(kp[0], kp[1]), pack_bf16(kp[2], kp[3]),
                                   pack_bf16(kp[4], kp[5]), pack_bf16(kp[6], kp[7]));
      st_s16(A1, kmajor_off(i, c0, 128), kpv);
      st_s16(B2, mnmajor_off(c0, i, kB2Sbo), kpv);
      st_s16(A1, kmajor_off(64 + i, c0, 128),
             make_uint4(pack_bf16(qp[0], qp[1]), pack_bf16(qp[2], qp[3]), pack_bf16(qp[4], qp[5]),
                        pack_bf16(qp[6], qp[7])));
      st_s16(B1, kmajor_off(i, c0, 64),
             make_uint4(pack_bf16(kn[0], kn[1]), pack_bf16(kn[2], kn[3]), pack_bf16(kn[4], kn[5]),
                        pack_bf16(kn[6], kn[7])));
      *reinterpret_cast<uint4*>(rec + Rec::AK + mnmajor_off(c0, i, Rec::kAkSbo)) =
          make_uint4(pack_bf16(kx[0], kx[1]), pack_bf16(kx[2], kx[3]), pack_bf16(kx[4], kx[5]),
                     pack_bf16(kx[6], kx[7]));
    }
    if (tb == 0) {  // every lane holds its channels' chunk totals
      float* gl = reinterpret_cast<float*>(rec + Rec::GL) + c0;
      *reinterpret_cast<float4*>(gl) = make_float4(GLm[0], GLm[1], GLm[2], GLm[3]);
      *reinterpret_cast<float4*>(gl + 4) = make_float4(GLm[4], GLm[5], GLm[6], GLm[7]);
    }

    // ---- the raw registers are free: the next item's rows are loaded in four
    // groups spread over this item's phases (g now, q, k, v below)
    const bool has_next = item + stride < n_items;
    const Chunk chn = ch_next;
    const int hn = (int)((item + stride) % H);
    if (has_next) load_part(p, chn, hn, tb, c0, 0, R.g);
    ch = ch_next;
    ch_next = item + 2 * stride < n_items ? p.chunks[(item + 2 * stride) / H] : Chunk{};

    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- MMA 1: [A_kk ; A_qk] = [Kp ; Qp] Kn^T   (M=128, N=64, K=128)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_bf16(tmem, sdesc(smem_u32(A1) + s * 2 * 128 * 16, 128 * 16, 128),
                 sdesc(smem_u32(B1) + s * 2 * 64 * 16, 64 * 16, 128), id, s > 0);
      mma_commit(&bar_mma);
    }
    if (has_next) load_part(p, chn, hn, tb, c0, 1, R.q);
    ok = __syncthreads_and(mbar_wait(&bar_mma, 0, kWaitLimitNs));
    fence_after_sync();
    if (!ok) break;
    {
      float d[32];
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + 32 * half;
      tmem_ld16(ta, d);
      tmem_ld16(ta + 16, d + 16);
      tmem_ld_wait();
      const int row = 32 * quarter + lane;
      if (quarter < 2) {
        const int i = row;
        const float bi = beta[i];
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          const int j = 32 * half + t;
          *reinterpret_cast<float4*>(AKK + i * kAs + j) =
              make_float4(j < i ? bi * d[t] : 0.f, j + 1 < i ? bi * d[t + 1] : 0.f,
                          j + 2 < i ? bi * d[t + 2] : 0.f, j + 3 < i ? bi * d[t + 3] : 0.f);
        }
      } else {
        const int i = row - 64;
        const bool live = i < len;
#pragma unroll
        for (int t8 = 0; t8 < 4; ++t8) {
          const int jb = 4 * half + t8;
          float a[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) a[t] = (live && 8 * jb + t <= i) ? d[8 * t8 + t] : 0.f;
          *reinterpret_cast<uint4*>(rec + Rec::AQ + kmajor_off(i, 8 * jb, 64)) =
              make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                         pack_bf16(a[6], a[7]));
        }
      }
    }
    if (has_next) load_part(p, chn, hn, tb, c0, 2, R.k);
    fence_before_sync();
    __syncthreads();

    // ---- T = (I + A_kk)^{-1}; Tb = T diag(beta) -> A2 (bf16, R=64)
    tri_inverse_64(AKK, TT, XS);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int idx = tid + kThreads * t;
      const int i = idx & 63, jb = idx >> 6;
      const float4 t0 = *reinterpret_cast<const float4*>(TT + i * kTs + 8 * jb);
      const float4 t1 = *reinterpret_cast<const float4*>(TT + i * kTs + 8 * jb + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(beta + 8 * jb);
      const float4 b1 = *reinterpret_cast<const float4*>(beta + 8 * jb + 4);
      st_s16(A2, kmajor_off(i, 8 * jb, 64),
             make_uint4(pack_bf16(t0.x * b0.x, t0.y * b0.y), pack_bf16(t0.z * b0.z, t0.w * b0.w),
                        pack_bf16(t1.x * b1.x, t1.y * b1.y), pack_bf16(t1.z * b1.z, t1.w * b1.w)));
    }
    if (has_next) {
      load_part(p, chn, hn, tb, c0, 3, R.v);
      R.b = load_b(p, chn, hn, tid);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    // ---- MMA 2: [W | U~] = Tb [Kp | V]   (M=64, N=256, K=64)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(64, 256, 0, 1);  // B2 is MN-major
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_bf16(tmem, sdesc(smem_u32(A2) + s * 2 * 64 * 16, 64 * 16, 128),
                 sdesc(smem_u32(B2) + s * 256, 128, kB2Sbo), id, s > 0);
      mma_commit(&bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma, 1, kWaitLimitNs));
    fence_after_sync();
    if (!ok) break;
    {
      // M=64 accumulator: row r sits in TMEM lane (r/16)*32 + r%16; warps 0-3
      // take W (columns 0-127), warps 4-7 take U~ (columns 128-255)
      const int i = 16 * quarter + (lane & 15);
      const bool row_lane = lane < 16;
      const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16) + 128 * half;
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        float d[32];
        tmem_ld16(ta + c, d);
        tmem_ld16(ta + c + 16, d + 16);
        tmem_ld_wait();
        if (row_lane) {
          if (half == 0) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              st_s16(A1, kmajor_off(i, c + 8 * u, 128),
                     make_uint4(pack_bf16(d[8 * u], d[8 * u + 1]), pack_bf16(d[8 * u + 2], d[8 * u + 3]),
                                pack_bf16(d[8 * u + 4], d[8 * u + 5]),
                                pack_bf16(d[8 * u + 6], d[8 * u + 7])));
          } else {
            float* ut = reinterpret_cast<float*>(rec + Rec::UT);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(ut + (((c >> 2) + q4) * 64 + i) * 4) =
                  make_float4(d[4 * q4], d[4 * q4 + 1], d[4 * q4 + 2], d[4 * q4 + 3]);
          }
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // [W ; Qp] to the record in one bulk copy; its completion is awaited
    // before A1 is rewritten by the next item
    if (tid == 0) {
      bulk_s2g(rec + Rec::AW, A1, 128 * 128 * 2);
      bulk_commit();
    }
  }
  if (tid == 0) {
    if (!ok) flag(p.status, kFlagTimeout);
    bulk_wait_all();
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

cudaError_t launch_intra(const ChunkParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tc_intra, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Smem::BYTES);
  if (e != cudaSuccess || p.max_chunks == 0) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t n_items = p.max_chunks * (int64_t)p.H;
  const int64_t grid = n_items < 2 * (int64_t)sms ? n_items : 2 * (int64_t)sms;
  tc_intra<<<(unsigned)grid, kThreads, Smem::BYTES, stream>>>(p, n_items);
  return cudaGetLastError();
}

}  // namespace tcp
}  // namespace kda
