// kda_tc_intra.cuh -- the intra-chunk step of the tensor-core prefill (K2)
// as a device function over one item pipeline, for the intra-chunk kernel
// (kda_tc_intra.cu, a pipeline per CTA) and the fused kernel (kda_tc_fused.cu,
// two pipelines per CTA beside the chain CTAs).
//
// A pipeline is 256 threads.  For each (chunk, head) item every thread owns 4 consecutive tokens x 8 channels: warp w takes channel
// half w % 2 and token quarter w / 2, lane l channel group l % 8 and token
// block l / 8.  A warp's 16-byte loads of one token row index then cover four
// whole 128-byte lines (coalesced); the rows are prefetched into L2 during
// the previous item.  The cumulative decay Gamma is a product scan (in
// registers over a thread's 4 tokens, across the warp's 4 token blocks with
// shuffles, across the 4 token quarters through shared memory), the norms
// reduce over 8 lanes and a pair of warps.  The operands are written with
// 16-byte shared stores straight into the tcgen05 no-swizzle layouts, whose
// stride between 8-channel groups is padded by 16 bytes so that the 8 channel
// groups and 4 tokens of one warp store fall in distinct banks.  Then:
//   MMA 1 (M=128, N=64, K=128):  [A_kk ; A_qk] = [Kp ; Qp] Kn^T  -> TMEM
//   CUDA cores: T = (I + A_kk)^{-1}, two-level blocked inverse
//   MMA 2 (M=64, N=256, K=64):   [W | U~] = T diag(beta) [Kp | V] -> TMEM
// and the record of kda_tc_common.cuh is written: AW and AK with bulk copies
// (TMA engine) out of shared memory, one per 8-channel group (dropping the
// padding), A_qk with one, each staged in a tile that is free at that point;
// U~ and Gamma_L with 16-byte stores.  The math is stated in
// kda_tc_common.cuh.
#pragma once

#include "kda_tc_handoff.cuh"

namespace kda {
namespace tcp {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kAs = 68;  // row stride (floats) of A_kk in shared memory
constexpr int kTs = 64;  // row stride (floats) of T
// Padded no-swizzle operand layouts (strides of the descriptors, bytes)
constexpr uint32_t kA1Lbo = 128 * 16 + 16;  // A1 K-major, R=128: stride between 8-channel groups
constexpr uint32_t kB1Lbo = 64 * 16 + 16;   // B1 K-major, R=64
constexpr uint32_t kB2Sbo = 8 * 128 + 16;   // B2 MN-major (n, token): stride between 8-n groups
constexpr uint32_t kA2Lbo = 64 * 16 + 16;   // A2 (T diag(beta)) K-major, R=64
constexpr uint32_t kAkStage = 8 * 128 + 16; // Kr^T staged for its record copy: stride between 8-channel groups
// threads that issue the record's bulk copies (each waits for its own).  The
// AW and AK copies go one per 8-channel group g, from lane g % 2 of warp
// g / 2: a bulk-copy issue holds its warp until the copy engine takes it, so
// spreading the 16 of a tile over the warps keeps any one warp from waiting
// for all of them.
constexpr int kAqCopy = 64;    // A_qk
__device__ __forceinline__ int copy_group(int tid) {
  return (tid & 31) < 2 ? 2 * (tid >> 5) + (tid & 31) : -1;
}
// threads that store rows of the record from registers: Gamma_L (warp 0)
// and U~ (lanes 0-15 of warps 4-7)
__device__ __forceinline__ bool writes_record_rows(int tid) {
  return tid < 32 || (tid >= 128 && (tid & 31) < 16);
}

struct Smem {
  static constexpr uint32_t A1 = 0;                    // [Kp;Qp] -> [W;Qp], K=128 (16 groups)
  static constexpr uint32_t B1 = A1 + 16 * kA1Lbo;     // Kn, K=128; then T fp32 [64][64]
  static constexpr uint32_t B2 = B1 + 16 * kB1Lbo;     // [Kp | V] MN-major, N=256 (32 groups), K=64
  static constexpr uint32_t A2 = B2 + 32 * kB2Sbo;     // inverse scratch; then Tb, R=64, K=64
  static constexpr uint32_t AKK = A2 + 8 * kA2Lbo;     // fp32 [64][kAs]
  // inv_q, inv_k, beta [64]; norm partials [q/k][channel half][64];
  // decay totals of each token quarter [4][128]
  static constexpr uint32_t MISC = AKK + 64 * kAs * 4;
  // + the per-token decay logits of the item (gate per head), [64]
  // + 2^s of each channel's decay reference and 2^(G_L - s) (see the
  // operands), [2][128]
  static constexpr uint32_t BYTES = MISC + (3 * 64 + 2 * 2 * 64 + 4 * 128 + 64 + 2 * 128) * 4;
};
static_assert(Smem::B1 % 16 == 0 && Smem::B2 % 16 == 0 && Smem::A2 % 16 == 0 && Smem::AKK % 16 == 0,
              "operand tiles and float4 arrays are 16-byte aligned");
static_assert(8 * kA2Lbo >= 64 * 64 * 2, "A2 holds the unpadded A_qk staging too");
static_assert(16 * kB1Lbo >= 64 * kTs * 4, "T fits in the Kn tile");
static_assert(32 * 40 * 4 <= 8 * kA2Lbo, "the inverse's product scratch fits in A2");
static_assert(16 * kAkStage <= 64 * kAs * 4, "the Kr^T staging fits in the A_kk tile");
static_assert(32 * kB2Sbo >= 64 * 128 * 4, "the U~ staging fits in the B2 tile");

// 8 floats from shared memory (16-byte aligned), read where the call stands
// (volatile: the compiler does not merge the reads of several calls, so it
// keeps no copy in registers between them).  The values are written before
// a barrier that precedes every call.
__device__ __forceinline__ void lds_f8(const float* p, float* x) {
  const uint32_t a = smem_u32(p);
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]) : "r"(a));
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]) : "r"(a + 16));
}
__device__ __forceinline__ void st_s16(uint8_t* base, uint32_t off, uint4 v) {
  *reinterpret_cast<uint4*>(base + off) = v;
}
// byte offset of element (r, k) of a K-major operand whose 8-channel groups
// are `lbo` bytes apart
__device__ __forceinline__ uint32_t kmaj(uint32_t r, uint32_t k, uint32_t lbo) {
  return (k >> 3) * lbo + (r >> 3) * 128u + (r & 7u) * 16u + (k & 7u) * 2u;
}

// T (64 x 64 fp32, row stride kTs) keeps its columns XOR-swizzled by row:
// element (r, c) at r kTs + (c ^ 8 (r % 4)).  Aligned groups of 8 columns
// stay contiguous (16-byte row reads are unchanged), and the 4 rows x 8
// columns that a warp-level MMA operand fragment reads fall in 32 distinct
// banks.
__device__ __forceinline__ int tsw(int r, int c) { return r * kTs + (c ^ ((r & 3) << 3)); }

// Warp-level tensor-core MMA, m16n8k8, tf32 operands, fp32 accumulator
// (d += a b): a = rows g, g+8 x columns t, t+4 of a 16 x 8 tile, b = rows t,
// t+4 x column g of an 8 x 8 tile, d = rows g, g+8 x columns 2t, 2t+1, with
// g = lane / 4 and t = lane % 4.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
constexpr int kXs = 40;  // row stride (floats) of the product scratch: 8 mod 32 banks

// One 16 x 8 tile of P = L R (K = 8 ks_n steps), L and R given as element
// readers: L(row, k) over rows m0 .. m0+15, R(k, col) over columns n0 .. n0+7.
template <int KS, typename LF, typename RF>
__device__ __forceinline__ void tile_product(float* d, int m0, int n0, int k0, LF L, RF R) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  d[0] = d[1] = d[2] = d[3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int k = k0 + 8 * ks + t;
    const uint32_t a[4] = {to_tf32(L(m0 + g, k)), to_tf32(L(m0 + g + 8, k)), to_tf32(L(m0 + g, k + 4)),
                           to_tf32(L(m0 + g + 8, k + 4))};
    const uint32_t b[2] = {to_tf32(R(k, n0 + g)), to_tf32(R(k + 4, n0 + g))};
    mma_tf32(d, a, b);
  }
}

// T = (I + A)^{-1} for strictly lower-triangular A (64x64, stride kAs).
// Level 0: the four 16x16 diagonal tiles by forward substitution (a thread
// per column, CUDA cores).  Level 1: the two 16x16 tiles below them inside
// each 32x32 half, T10 = -T11 A10 T00.  Level 2: the lower-left 32x32 tile,
// T = -T_hi A T_lo.  The products of levels 1 and 2 run on the warp-level
// tensor cores in tf32 with fp32 accumulation (T is rounded to bf16 once
// scaled by beta, far coarser than tf32).  X: scratch of 32 x kXs floats.
// The 256 threads of one item pipeline (tid 0..255, barrier bs); the thread
// given x_busy first waits until its bulk copy out of X has read it.
__device__ __forceinline__ void tri_inverse_64(const float* __restrict__ A, float* __restrict__ T,
                                               float* __restrict__ X, bool x_busy, int tid,
                                               const PipeSync& bs) {
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
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
    for (int ii = 0; ii < 16; ++ii) T[tsw(16 * d + ii, j)] = col[ii];
  } else {
    // tiles strictly above the diagonal are zero
    for (int idx = tid - 64; idx < 6 * 256; idx += kThreads - 64) {
      const int tt = idx >> 8, e = idx & 255;
      const int bi = tt < 3 ? 0 : (tt < 5 ? 1 : 2);
      const int bj = tt < 3 ? tt + 1 : (tt < 5 ? tt - 1 : 3);
      T[tsw(16 * bi + (e >> 4), 16 * bj + (e & 15))] = 0.f;
    }
  }
  if (x_busy) bulk_wait_read_all();
  bs.sync();
  // level 1, warps 0-3: P = warp / 2 -> tile rows r0 = 32P+16.., cols c0 = 32P..,
  // 8-column half warp % 2.  (X held the staged A_qk of the record: its copy
  // has read it.)
  auto Ael = [&](int r, int c) { return A[r * kAs + c]; };
  auto Tel = [&](int r, int c) { return T[tsw(r, c)]; };
  const int P = warp >> 1, nh = warp & 1, r0 = 32 * P + 16, c0 = 32 * P;
  float* X1 = X + P * 16 * kXs;
  float d[4];
  if (warp < 4) {
    tile_product<2>(d, r0, c0 + 8 * nh, c0, Ael, Tel);  // A10 T00
    const int c = 8 * nh + 2 * t;
    X1[g * kXs + c] = d[0];
    X1[g * kXs + c + 1] = d[1];
    X1[(g + 8) * kXs + c] = d[2];
    X1[(g + 8) * kXs + c + 1] = d[3];
  }
  bs.sync();
  if (warp < 4) {
    auto Xel = [&](int r, int c) { return X1[(r - r0) * kXs + c - c0]; };
    tile_product<2>(d, r0, c0 + 8 * nh, r0, Tel, Xel);  // T11 (A10 T00)
    const int c = c0 + 8 * nh + 2 * t;
    T[tsw(r0 + g, c)] = -d[0];
    T[tsw(r0 + g, c + 1)] = -d[1];
    T[tsw(r0 + g + 8, c)] = -d[2];
    T[tsw(r0 + g + 8, c + 1)] = -d[3];
  }
  bs.sync();
  // level 2, all warps: rows 32..63, cols 0..31; warp w takes rows 32 + 16 (w / 4)..,
  // columns 8 (w % 4)..
  {
    const int m0 = 32 + 16 * (warp >> 2), n0 = 8 * (warp & 3);
    tile_product<4>(d, m0, n0, 0, Ael, Tel);  // A[32:64, 0:32] T[0:32, 0:32]
    const int r = m0 - 32 + g, c = n0 + 2 * t;
    X[r * kXs + c] = d[0];
    X[r * kXs + c + 1] = d[1];
    X[(r + 8) * kXs + c] = d[2];
    X[(r + 8) * kXs + c + 1] = d[3];
    bs.sync();
    auto Xel = [&](int rr, int cc) { return X[(rr - 32) * kXs + cc]; };
    tile_product<4>(d, m0, n0, 32, Tel, Xel);  // T[32:64, 32:64] X
    T[tsw(m0 + g, c)] = -d[0];
    T[tsw(m0 + g, c + 1)] = -d[1];
    T[tsw(m0 + g + 8, c)] = -d[2];
    T[tsw(m0 + g + 8, c + 1)] = -d[3];
  }
  bs.sync();
}

// The raw rows of an item are staged row-major ([64 tokens][128 channels]
// bf16, 256 bytes a row) by one tensor-map copy per tensor (TMA engine: box
// of 128 channels x 1 head x 64 tokens), inside operand tiles that are free
// at that point: g in B1 and k in the A_kk tile (group A, once T diag(beta)
// is formed), q and v in B2 (group B, once MMA 2 has read it).  Every thread
// reads its raw chunks into registers before the first barrier of the item
// and writes operands over the staging only after the second.  Rows past the
// chunk's length hold other tokens (or zeros past the tensor's end) and are
// masked where they are read.
constexpr uint32_t kGStage = Smem::B1, kKStage = Smem::AKK, kQStage = Smem::B2,
                   kVStage = Smem::B2 + 64 * 256;
static_assert(16 * kB1Lbo >= 64 * 256 && 64 * kAs * 4 >= 64 * 256 && 32 * kB2Sbo >= 2 * 64 * 256,
              "the staging fits the tiles it borrows");
static_assert(kGStage % 128 == 0 && kKStage % 128 == 0 && kQStage % 128 == 0 && kVStage % 128 == 0,
              "tensor-map copies land on 128-byte boundaries");
constexpr uint32_t kRowsBytes = 64 * 256;  // one tensor's rows of an item

// Tensor maps of q, k, v, g viewed as [T][H][128] bf16, box {128, 1, 64};
// with the short convolution also q, k, v with box {128, 1, 3}: the halo
// rows, the three tokens before an item's first (a negative start reads
// zeros)
struct RowMaps {
  CUtensorMap g, q, k, v;
  CUtensorMap qh, kh, vh;
};

// The halo rows of the short convolution ("Kimi K3: The Manos, The Mythos,
// The Legendos", bullet on the stability details), KDA_CONV_MAX - 1 rows of
// 256 bytes per tensor, staged with their tensor's group in tiles that are
// free from the staging to the raw reads: k's after its rows in the A_kk
// tile (group A), q's and v's in A2 (group B, issued once MMA 2 has read A2;
// A2 is next written after MMA 1 of the item).
constexpr int kHaloRows = KDA_CONV_MAX - 1;
constexpr uint32_t kHaloBytes = kHaloRows * 256;
constexpr uint32_t kKHalo = kKStage + kRowsBytes, kQHalo = Smem::A2, kVHalo = Smem::A2 + kHaloBytes;
static_assert(kKHalo + kHaloBytes <= Smem::AKK + 64 * kAs * 4 && 2 * kHaloBytes <= 8 * kA2Lbo,
              "the halo rows fit the tiles they borrow");
static_assert(kKHalo % 128 == 0 && kQHalo % 128 == 0 && kVHalo % 128 == 0,
              "halo copies land on 128-byte boundaries");
// The convolution's taps of the item's head (fp32, 128 channels a tap),
// staged with group B after the q and v halo rows: tap j of tensor t at
// kWStage + (4 t + j) * 512.  L1 holds little beside the shared memory, so
// reading them from global memory would wait on L2 every item.
constexpr uint32_t kTapBytes = kD * 4;
constexpr uint32_t kWStage = kVHalo + kHaloBytes;
static_assert(kWStage + 3 * KDA_CONV_MAX * kTapBytes <= Smem::A2 + 8 * kA2Lbo && kWStage % 128 == 0,
              "the taps fit in A2 after the halo rows");

// rows of one tensor, tokens tok0..tok0+63 of head h, into shared memory
__device__ __forceinline__ void tma_rows(uint8_t* dst, const CUtensorMap* m, int h, int tok0,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(m), "r"(0), "r"(h), "r"(tok0), "r"(smem_u32(bar))
      : "memory");
}
// the same rows into L2 only
__device__ __forceinline__ void tma_rows_l2(const CUtensorMap* m, int h, int tok0) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(m), "r"(0), "r"(h),
               "r"(tok0)
               : "memory");
}

// What an item needs of its chunk-table entry: first token and length (the
// token index fits the int32 coordinates of the tensor maps on this path);
// with the short convolution also, packed as 4 seq + pre, how many of the
// halo rows lie inside the sequence (pre, at most kHaloRows) and the
// sequence (for its window).  A few registers instead of the entry's eight.
struct ItemChunk {
  int tok0, len, aux;
  __device__ __forceinline__ int pre() const { return aux & 3; }
  __device__ __forceinline__ int seq() const { return aux >> 2; }
};
static_assert(kHaloRows <= 3, "pre fits two bits");
template <bool kConv>
__device__ __forceinline__ ItemChunk item_chunk(const ChunkParams& p, int64_t idx) {
  const Chunk* c = p.chunks + idx;
  ItemChunk r{(int)c->tok0, c->len, 0};
  if (kConv) {
    // segment scan: the table's sequences are segments of sequence 0, which
    // starts at token 0
    const int64_t pos = p.conv_one_seq ? c->tok0 : c->pos;
    const int seq = p.conv_one_seq ? 0 : c->seq;
    r.aux = 4 * seq + (pos < kHaloRows ? (int)pos : kHaloRows);
  }
  return r;
}

// Staging group A of item (ch, h): the rows of g (not with a gate per head)
// and k, and k's halo rows with the convolution, counted on `bar`.  Issued
// by one thread.
template <bool kHeadGate, bool kConv>
__device__ __forceinline__ void stage_a(uint8_t* sm, uint64_t* bar, const ItemChunk& ch, int h,
                                        const RowMaps& maps) {
  mbar_arrive_expect_tx(bar, (kHeadGate ? 1 : 2) * kRowsBytes + (kConv ? kHaloBytes : 0));
  if (!kHeadGate) tma_rows(sm + kGStage, &maps.g, h, ch.tok0, bar);
  tma_rows(sm + kKStage, &maps.k, h, ch.tok0, bar);
  if (kConv) tma_rows(sm + kKHalo, &maps.kh, h, ch.tok0 - kHaloRows, bar);
}

// Staging group B of item (ch, h): the rows of q and v (and, with the
// convolution, their halo rows and head h's taps).
template <bool kConv>
__device__ __forceinline__ void stage_b(uint8_t* sm, uint64_t* bar, const ItemChunk& ch, int h,
                                        const RowMaps& maps, const ChunkParams& p) {
  const int W = kConv ? p.conv_width : 0;
  mbar_arrive_expect_tx(bar, 2 * kRowsBytes + (kConv ? 2 * kHaloBytes + 3 * W * kTapBytes : 0));
  tma_rows(sm + kQStage, &maps.q, h, ch.tok0, bar);
  tma_rows(sm + kVStage, &maps.v, h, ch.tok0, bar);
  if (kConv) {
    tma_rows(sm + kQHalo, &maps.qh, h, ch.tok0 - kHaloRows, bar);
    tma_rows(sm + kVHalo, &maps.vh, h, ch.tok0 - kHaloRows, bar);
    for (int t = 0; t < 3; ++t)
      for (int j = 0; j < W; ++j)
        bulk_g2s(sm + kWStage + (4 * t + j) * kTapBytes, p.conv_w[t] + ((size_t)j * p.H + h) * kD, kTapBytes,
                 bar);
  }
}

// 16 bytes of a raw row in a staging: token i, channels c0..c0+7
__device__ __forceinline__ uint4 raw16(const uint8_t* sm, uint32_t stage, int i, int c0) {
  return *reinterpret_cast<const uint4*>(sm + stage + i * 256 + c0 * 2);
}

// 16 bytes of input row -back (back = 1..kHaloRows tokens before the item's
// first) of one tensor: the staged halo row while inside the sequence, else
// the sequence's window row (W - 1) - (tokens before the sequence start), or
// zeros without a window; zeros past the convolution's reach
__device__ __forceinline__ uint4 halo16(const uint8_t* sm, uint32_t halo, const void* win,
                                        const ChunkParams& p, const ItemChunk& ch, int h, int back, int c0) {
  const int W = p.conv_width;
  if (back > W - 1) return make_uint4(0, 0, 0, 0);
  if (back <= ch.pre()) return raw16(sm, halo, kHaloRows - back, c0);
  if (!win) return make_uint4(0, 0, 0, 0);
  const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(win);
  const int64_t row = (int64_t)ch.seq() * (W - 1) + (W - 1) - (back - ch.pre());
  return *reinterpret_cast<const uint4*>(wb + (row * p.H + h) * kD + c0);
}

// Rows i0..i0+3 (channels c0..c0+7) of tensor t (0 q, 1 k, 2 v) after the
// short convolution, as bf16: y_i = sum_{j < W} w[j][h][c] x_{i-j} (taps at
// or past W count as 0), SiLU if asked (silu_fast), rounded to bf16 (the input dtype);
// rows at or past len give zeros, as the raw rows do.  The inputs come from
// the item's staging and, for the first token block, the halo; the taps
// from their staging.
__device__ __forceinline__ void conv_rows(const uint8_t* sm, uint32_t stage, uint32_t halo, int t,
                                          const ChunkParams& p, const ItemChunk& ch, int h, int i0, int c0,
                                          uint4 out[4]) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  uint4 x[7];  // input rows i0 - 3 .. i0 + 3
#pragma unroll
  for (int m = 0; m < 7; ++m) {
    const int i = i0 - kHaloRows + m;
    x[m] = i >= 0 ? (i < ch.len ? raw16(sm, stage, i, c0) : z) : halo16(sm, halo, p.conv_in[t], p, ch, h, -i, c0);
  }
  const int W = p.conv_width;
  const float* w = reinterpret_cast<const float*>(sm + kWStage + 4 * t * kTapBytes) + c0;  // staged taps
  uint32_t o[4][4];
#pragma unroll
  for (int pp = 0; pp < 4; ++pp) {  // channel pair c0 + 2 pp, c0 + 2 pp + 1, two lanes of f32x2
    float2 wv[4], xv[7];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      wv[j] = j < W ? *reinterpret_cast<const float2*>(w + j * kD + 2 * pp) : make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < 7; ++m) {
      const uint32_t wd = pp == 0 ? x[m].x : pp == 1 ? x[m].y : pp == 2 ? x[m].z : x[m].w;
      xv[m] = make_float2(bf16_lo(wd), bf16_hi(wd));
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float2 a = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 4; ++j) a = __ffma2_rn(wv[j], xv[r + kHaloRows - j], a);
      if (p.conv_silu) {
        a.x = silu_fast(a.x);
        a.y = silu_fast(a.y);
      }
      o[r][pp] = i0 + r < ch.len ? pack_bf16(a.x, a.y) : 0u;
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) out[r] = make_uint4(o[r][0], o[r][1], o[r][2], o[r][3]);
}

__device__ __forceinline__ float load_b(const ChunkParams& p, const ItemChunk& ch, int h, int tid) {
  const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(p.b);
  return (tid < 64 && tid < ch.len) ? __bfloat162float(gb[((int64_t)ch.tok0 + tid) * p.H + h]) : 0.f;
}
// the decay logit of token tid of item (ch, h) with a gate per head (g [T, H]);
// rows past the chunk get 0 (they are masked where they are used)
__device__ __forceinline__ float load_gh(const ChunkParams& p, const ItemChunk& ch, int h, int tid) {
  const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(p.g);
  return (tid < 64 && tid < ch.len) ? __bfloat162float(gg[((int64_t)ch.tok0 + tid) * p.H + h]) : 0.f;
}

// The mbarriers of one item pipeline, and the outcome of its wait for a
// free slot of the record ring
struct IntraBars {
  uint64_t mma;
  uint64_t ga, gb;  // staging groups A (g, k) and B (q, v)
  uint64_t drain;   // every MMA, on the error path
  // (thread 0) the flags of this item's record and of the record that is
  // complete but not yet published (or null)
  uint32_t* cur;
  uint32_t* pend;
  // (items taken from the shared counter) the pipeline's coming items: item
  // n + k of the pipeline (k = 1..3 ahead of item n) in entry (n + k) % 4;
  // thread 0 takes item n + 3 during item n.  `stopped`: a pipeline that
  // leaves at the split has taken its last item
  int64_t ahead[4];
  int32_t stopped;
};
__device__ __forceinline__ void init_intra_bars(IntraBars* b) {
  mbar_init(&b->mma, 1);
  mbar_init(&b->ga, 1);
  mbar_init(&b->gb, 1);
  mbar_init(&b->drain, 1);
  mbar_init_fence();
  b->pend = nullptr;
  b->stopped = 0;
}

// One item pipeline: 256 threads (tid 0..255) on Smem::BYTES of shared
// memory at sm, 256 TMEM columns at tmem, synchronised by bs; it takes the
// items first, first + stride, ... below n_items (or, with items taken from
// the overlapped schedule's counter, those it takes there; `stay`: it takes
// items until none is left, else only while fewer than p.ovl_split have
// been taken).
struct IntraPipe {
  uint8_t* sm;
  IntraBars* bars;
  uint32_t tmem;
  int tid;
  PipeSync bs;
  int64_t first, stride, n_items;
  bool stay;
};

// (thread 0, overlapped schedule) the next item of this pipeline from the
// shared counter, or INT64_MAX for none.  Items are taken in index order,
// that is in chunk order, the order in which the chains read them.  A
// pipeline that leaves at the split takes no more items once it has taken
// one at or past the split (which it still makes).
__device__ __forceinline__ int64_t take_item(const ChunkParams& p, const IntraPipe& x) {
  if (x.bars->stopped) return INT64_MAX;
  const unsigned long long i = atomicAdd(&p.ovl->next_item, 1ull);
  if (!x.stay && i >= (unsigned long long)p.ovl_split) x.bars->stopped = 1;
  return i < (unsigned long long)x.n_items ? (int64_t)i : INT64_MAX;
}

// The items of one pipeline.  The next item's rows are prefetched into L2 at
// the top of an item and staged by bulk copies as soon as their tiles are
// free.  TMEM and the mbarriers are set up by the caller.
// kPoll: the instantiation for wait limits under kPollLimitNs (the give-up
// test).  kHeadGate: g is [T, H], one decay per token and head (the gated
// delta rule): no g rows are staged, the scan runs over tokens only.
// kConv: q, k, v pass through the short convolution as they are read.
// kFused: the chains of the fused kernel read the records as they come: the
// record of each item is published (kda_tc_handoff.cuh) once its copies
// have landed, at a barrier of the pipeline's next item (or after its last).
// kTake: the items come from the overlapped schedule's counter (take_item)
// instead of a stride; each is known three items ahead of its turn, as the
// prefetches need.
template <bool kPoll, bool kHeadGate, bool kConv, bool kFused, bool kTake = false>
__device__ __forceinline__ void intra_items(const ChunkParams& p, const RowMaps& maps, const IntraPipe& x) {
  uint8_t* const sm = x.sm;
  uint64_t& bar_mma = x.bars->mma;
  uint64_t& bar_ga = x.bars->ga;
  uint64_t& bar_gb = x.bars->gb;
  uint64_t& bar_drain = x.bars->drain;
  const PipeSync bs = x.bs;
  const int64_t stride = x.stride, n_items = x.n_items;
  int64_t item = x.first;
  const int H = p.H;
  const int tid = x.tid, warp = tid >> 5, lane = tid & 31;
  // this thread: tokens i0 .. i0 + 3, channels c0 .. c0 + 7
  const int cg = lane & 7, tb = lane >> 3;  // channel group in the half, token block in the quarter
  const int hc = warp & 1, qt = warp >> 1;  // channel half, token quarter
  const int c0 = 64 * hc + 8 * cg;
  const int i0 = 16 * qt + 4 * tb;
  // TMEM lane quarter and column half, for the accumulator read-outs
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
  float* nrm = beta + 64;        // [q/k][channel half][64]
  float* qtot = nrm + 2 * 2 * 64;  // [token quarter][128]
  float* gtok = qtot + 4 * 128;    // [64] decay logits of this item's tokens (gate per head)
  float* sref = gtok + 64;         // [128] 2^s per channel (decay reference)
  float* sglr = sref + 128;        // [128] 2^(G_L - s) per channel

  // the pipeline: chunk entries of the current and the next item; the first
  // item's rows are staged here (groups A and B), each later item's during
  // the item before it
  // (chunk-table entries are read two items ahead of their first use, the
  // L2 prefetch of the next item's rows: a global load's latency is hidden)
  // the pipeline's item k ahead of its n-th (INT64_MAX or past n_items: none)
  int64_t* const ahead = x.bars->ahead;
  auto item_ahead = [&](uint32_t n, int k) -> int64_t {
    return kTake ? ahead[(n + k) & 3] : item + k * stride;
  };
  if constexpr (kTake) {
    if (tid == 0) {
      item = take_item(p, x);
      for (int k = 1; k <= 2; ++k) ahead[k] = take_item(p, x);
      ahead[0] = item;
    }
    bs.sync();
    item = ahead[0];
    if (item >= n_items) return;  // (uniform) nothing left: no staging was issued
  }
  ItemChunk ch = item_chunk<kConv>(p, item / H);  // entries past the table's end have len 0
  ItemChunk ch_next = item_ahead(0, 1) < n_items ? item_chunk<kConv>(p, item_ahead(0, 1) / H) : ItemChunk{0, 0, 0};
  ItemChunk ch_next2 = item_ahead(0, 2) < n_items ? item_chunk<kConv>(p, item_ahead(0, 2) / H) : ItemChunk{0, 0, 0};
  {
    const int h0 = (int)(item % H);
    if (tid == 0) {
      stage_a<kHeadGate, kConv>(sm, &bar_ga, ch, h0, maps);
      stage_b<kConv>(sm, &bar_gb, ch, h0, maps, p);
    }
    if (kHeadGate && tid < 64) gtok[tid] = load_gh(p, ch, h0, tid);
  }
  bool a_fly = true, b_fly = true;  // staging groups in flight, not yet awaited
  uint32_t sph = 0;                 // the phase they complete
  float bnext = load_b(p, ch, (int)(item % H), tid);
  float gnext = 0.f;                // the next item's decay logit of token tid (gate per head)

  fence_before_sync();
  bs.sync();
  fence_after_sync();
  const uint32_t tmem = x.tmem;
  bool ok = true;

  uint32_t nth = 0;  // (kTake) the pipeline's count of items so far
  for (; item < n_items;) {
    const int h = (int)(item % H);
    const int64_t cidx = item / H;
    const int len = ch.len;

    // past the end of the chunk table (uniform across the CTA); every later
    // item of this CTA is past it too
    if (len == 0) break;
    uint8_t* rec = reinterpret_cast<uint8_t*>(p.inter) + ((size_t)cidx * H + h) * Rec::BYTES;
    if (kFused && tid == 0) x.bars->cur = rec_flag(p, cidx, h);
    const int64_t item1 = item_ahead(nth, 1);
    const bool has_next = item1 < n_items;
    const ItemChunk chn = ch_next;
    const int hn = has_next ? (int)(item1 % H) : 0;
    const float bcur = bnext;
    // the next item's rows into L2 now, so that their staging copies hit L2
    if (has_next && tid < 4 && !(kHeadGate && tid == 0))
      tma_rows_l2(tid == 0 ? &maps.g : tid == 1 ? &maps.k : tid == 2 ? &maps.q : &maps.v, hn,
                  chn.tok0);
    // this item's g and k (group A) have landed; q and v (group B) may still fly
    ok = mbar_wait_t<kPoll>(&bar_ga, sph, p.wait_ns);
    a_fly = false;
    if constexpr (kConv) {
      // the convolution, before the decay scan: q and v (group B) were staged
      // during the previous item.  Its results replace the staged rows (once
      // every thread has read its inputs, some of them other threads' rows),
      // and the raw reads below take them from there like unconvolved rows:
      // no registers are held through the scan.
      ok = mbar_wait_t<kPoll>(&bar_gb, sph, p.wait_ns) && ok;
      b_fly = false;
      // one tensor at a time (a barrier each): only its 16 registers of
      // results are live
#pragma unroll 1
      for (int u = 0; u < 3; ++u) {  // k (tensor 1), q (0), v (2)
        const uint32_t stage = u == 0 ? kKStage : u == 1 ? kQStage : kVStage;
        const uint32_t halo = u == 0 ? kKHalo : u == 1 ? kQHalo : kVHalo;
        uint4 y[4];
        conv_rows(sm, stage, halo, u == 0 ? 1 : u == 1 ? 0 : 2, p, ch, h, i0, c0, y);
        bs.sync();
#pragma unroll
        for (int r = 0; r < 4; ++r) st_s16(sm, stage + (i0 + r) * 256 + c0 * 2, y[r]);
      }
    }

    // ---- cumulative decay G_i = sum_{m<=i} log2 alpha_m (alpha = exp(-softplus(g)),
    // log2 units): a sum over this thread's 4 tokens, a scan across the
    // warp's 4 token blocks (lanes 8 apart), then across the token quarters
    // through shared memory (below).  In log space G does not underflow,
    // whatever the decay.
    float Gm[4][8], qtot_own[8];
    // the scan of one channel: a[r] = log2 alpha of token i0 + r -> Gm[r][j], qtot_own[j]
    auto scan_channel = [&](const float* a, int j) {
      float run = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        run += a[r];
        Gm[r][j] = run;
      }
      float inc = run;
      float y = __shfl_up_sync(0xffffffffu, inc, 8);
      if (tb >= 1) inc += y;
      y = __shfl_up_sync(0xffffffffu, inc, 16);
      if (tb >= 2) inc += y;
      float ex = __shfl_up_sync(0xffffffffu, inc, 8);
      if (tb == 0) ex = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) Gm[r][j] += ex;
      qtot_own[j] = __shfl_sync(0xffffffffu, inc, 24 + cg);  // this quarter's sum
    };
    if constexpr (kHeadGate) {
      // one decay per token: the scan of one channel, shared by all eight
      float a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = i0 + r < len ? log2_alpha_fast(gtok[i0 + r]) : 0.f;
      scan_channel(a, 0);
#pragma unroll
      for (int j = 1; j < 8; ++j) {
        qtot_own[j] = qtot_own[0];
#pragma unroll
        for (int r = 0; r < 4; ++r) Gm[r][j] = Gm[r][0];
      }
    } else {
      uint4 graw[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) graw[r] = raw16(sm, kGStage, i0 + r, c0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float a[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = i0 + r < len ? log2_alpha_fast(bf16_at(graw[r], j)) : 0.f;
        scan_channel(a, j);
      }
    }
    if (tb == 0) {
      *reinterpret_cast<float4*>(qtot + qt * 128 + c0) =
          make_float4(qtot_own[0], qtot_own[1], qtot_own[2], qtot_own[3]);
      *reinterpret_cast<float4*>(qtot + qt * 128 + c0 + 4) =
          make_float4(qtot_own[4], qtot_own[5], qtot_own[6], qtot_own[7]);
    }

    // ---- L2 norms per token: 8 channels here, 8 lanes, then the two channel
    // halves.  The raw q, k, v chunks go to registers now: the operands are
    // written over their stagings after the next two barriers.
    if constexpr (!kConv) {
      ok = mbar_wait_t<kPoll>(&bar_gb, sph, p.wait_ns) && ok;
      b_fly = false;
    }
    sph ^= 1;
    // (each thread reads back exactly the rows and channels it convolved)
    uint4 qraw[4], kraw[4], vraw[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const bool live = i0 + r < len;
      const uint4 z = make_uint4(0, 0, 0, 0);
      qraw[r] = live ? raw16(sm, kQStage, i0 + r, c0) : z;
      kraw[r] = live ? raw16(sm, kKStage, i0 + r, c0) : z;
      vraw[r] = live ? raw16(sm, kVStage, i0 + r, c0) : z;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float xq = bf16_at(qraw[r], j), xk = bf16_at(kraw[r], j);
        sq += xq * xq;
        sk += xk * xk;
      }
#pragma unroll
      for (int m = 1; m < 8; m <<= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, m);
        sk += __shfl_xor_sync(0xffffffffu, sk, m);
      }
      if (cg == 0) {
        nrm[hc * 64 + i0 + r] = sq;
        nrm[128 + hc * 64 + i0 + r] = sk;
      }
    }
    // beta = sigmoid(b) with the fast exponential and division (it enters
    // T diag(beta), which is rounded to bf16)
    if (tid < 64) beta[tid] = tid < len ? __fdividef(1.f, 1.f + __expf(-bcur)) : 0.f;
    // the previous item's record copies must have read A1 before it is
    // rewritten; in the fused kernel they must have landed (the record is
    // published below), and so must its U~ and Gamma_L stores
    if constexpr (kFused) {
      if (copy_group(tid) >= 0) {
        bulk_wait_all();
        fence_proxy_async_global();
      }
      if (writes_record_rows(tid)) fence_gpu();
    } else {
      if (copy_group(tid) >= 0) bulk_wait_read_all();
    }
    ok = bs.all(ok);
    if (!ok) {
      // a wait above gave up: this item's staging groups may still be in
      // flight; mark both, with their phase, for the drain at the end
      a_fly = b_fly = true;
      sph ^= 1;
      break;
    }
    if (kFused && tid == 0 && x.bars->pend) {
      // the previous record: its copies and stores landed before the barrier
      st_release_u32(x.bars->pend, 1u);
      x.bars->pend = nullptr;
    }
    if (tid < 64) {
      // 1 / max(|x|, 1e-6) = rsqrt(max(|x|^2, 1e-12)), with the hardware
      // reciprocal square root (the operands it scales are rounded to bf16)
      inv_q[tid] = rsqrtf(fmaxf(nrm[tid] + nrm[64 + tid], 1e-12f));
      inv_k[tid] = rsqrtf(fmaxf(nrm[128 + tid] + nrm[192 + tid], 1e-12f));
    }
    // ---- V into B2 MN-major rows 128..255 (every raw row has been read:
    // the staging is free): the raw 16 bytes are one core-matrix row
#pragma unroll
    for (int r = 0; r < 4; ++r) st_s16(B2, mnmajor_off(128 + c0, i0 + r, kB2Sbo), vraw[r]);
    // the decay entering this token quarter, and the chunk total G_L; then
    // per channel the reference s, 2^s and 2^(G_L - s); Gm becomes t = G - s.
    // s = 0 while G_L >= -kScaleFromLog2 (the factors 2^G and 2^-G of a
    // chunk-start reference are then normal); past that s = round(G_L / 2),
    // clamped so that 2^s stays normal
    float two_s[8], glr[8];
    bool rescale = false;  // some channel of this item has s != 0
    {
      float pre[8], tot[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) pre[j] = tot[j] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = *reinterpret_cast<const float4*>(qtot + q * 128 + c0);
        const float4 b = *reinterpret_cast<const float4*>(qtot + q * 128 + c0 + 4);
        const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (q < qt) pre[j] += x[j];
          tot[j] += x[j];
        }
      }
      bool out_of_range = false;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        out_of_range |= tot[j] < -kMaxChunkDecayLog2;
        const float sj = tot[j] < -kScaleFromLog2 ? fmaxf(rintf(0.5f * tot[j]), -126.f) : 0.f;
        rescale |= sj != 0.f;
        two_s[j] = __int_as_float(((int)sj + 127) << 23);
        glr[j] = exp2_fast(tot[j] - sj);
#pragma unroll
        for (int r = 0; r < 4; ++r) Gm[r][j] += pre[j] - sj;
      }
      // warps 0 and 1 hold every channel's total (uniform per warp)
      if (qt == 0 && __any_sync(0xffffffffu, out_of_range) && lane == 0) flag(p.status, kFlagDecayRange);
      if (qt == 0 && tb == 0) {  // warps 0-1, lanes 0-7: Gamma_L and 2^s of all 128 channels
        *reinterpret_cast<float4*>(sref + c0) = make_float4(two_s[0], two_s[1], two_s[2], two_s[3]);
        *reinterpret_cast<float4*>(sref + c0 + 4) = make_float4(two_s[4], two_s[5], two_s[6], two_s[7]);
        *reinterpret_cast<float4*>(sglr + c0) = make_float4(glr[0], glr[1], glr[2], glr[3]);
        *reinterpret_cast<float4*>(sglr + c0 + 4) = make_float4(glr[4], glr[5], glr[6], glr[7]);
      }
    }
    rescale = bs.any(rescale);
    // Gamma_L of the record, from the values in shared memory
    if (tid < 32) {
      const float4 s = *reinterpret_cast<const float4*>(sref + 4 * tid);
      const float4 gq = *reinterpret_cast<const float4*>(sglr + 4 * tid);
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(rec + Rec::GL) + 4 * tid) =
          make_float4(gq.x * s.x, gq.y * s.y, gq.z * s.z, gq.w * s.w);
    }

    // ---- operands.  With a = 2^t (t = G - s): MMA 1 takes Kp' = k^ a, Qp' =
    // q^ a (A1) and Kn' = k^ / a (B1), whose products are those of Kp Kn^T
    // and Qp Kn^T (the 2^s cancel) with every factor inside the normal range;
    // MMA 2 takes Kp = k^ Gamma (B2 MN-major rows 0-127, Gamma = a 2^s) and
    // the record Kr = k^ Gamma_L / Gamma = Kn' 2^(G_L - s) (staged MN-major
    // in the A_kk tile for the record's AK).  The record's Qp = q^ Gamma is
    // Qp' 2^s: where some s != 0, A1's rows 64-127 are scaled by 2^s once
    // MMA 1 has read them (an exact power-of-two scaling)
    uint8_t* AKS = sm + Smem::AKK;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = i0 + r;
      const float ik = inv_k[i], iq = inv_q[i];
      const uint4 qr = qraw[r], kr = kraw[r];
      // the channels' 2^s and 2^(G_L - s), re-read for every row (kept out of
      // registers across the loop)
      float ts[8], tg[8];
      lds_f8(sref + c0, ts);
      lds_f8(sglr + c0, tg);
      float kp[8], ks[8], qs[8], kn[8], kx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float kh = bf16_at(kr, j) * ik;
        const float qh = bf16_at(qr, j) * iq;
        const float a = exp2_fast(Gm[r][j]);
        ks[j] = kh * a;
        qs[j] = qh * a;
        kp[j] = ks[j] * ts[j];
        kn[j] = kh * exp2_fast(-Gm[r][j]);
        kx[j] = kn[j] * tg[j];
      }
      st_s16(A1, kmaj(i, c0, kA1Lbo),
             make_uint4(pack_bf16(ks[0], ks[1]), pack_bf16(ks[2], ks[3]), pack_bf16(ks[4], ks[5]),
                        pack_bf16(ks[6], ks[7])));
      st_s16(B2, mnmajor_off(c0, i, kB2Sbo),
             make_uint4(pack_bf16(kp[0], kp[1]), pack_bf16(kp[2], kp[3]), pack_bf16(kp[4], kp[5]),
                        pack_bf16(kp[6], kp[7])));
      st_s16(A1, kmaj(64 + i, c0, kA1Lbo),
             make_uint4(pack_bf16(qs[0], qs[1]), pack_bf16(qs[2], qs[3]), pack_bf16(qs[4], qs[5]),
                        pack_bf16(qs[6], qs[7])));
      st_s16(B1, kmaj(i, c0, kB1Lbo),
             make_uint4(pack_bf16(kn[0], kn[1]), pack_bf16(kn[2], kn[3]), pack_bf16(kn[4], kn[5]),
                        pack_bf16(kn[6], kn[7])));
      st_s16(AKS, mnmajor_off(c0, i, kAkStage),
             make_uint4(pack_bf16(kx[0], kx[1]), pack_bf16(kx[2], kx[3]), pack_bf16(kx[4], kx[5]),
                        pack_bf16(kx[6], kx[7])));
    }

    fence_async_smem();
    fence_before_sync();
    bs.sync();
    fence_after_sync();

    // Kr^T to the record's AK, one bulk copy per 8-channel group (dropping
    // the staging's padding)
    if (copy_group(tid) >= 0) {
      const int g = copy_group(tid);
      bulk_s2g(rec + Rec::AK + g * Rec::kAkSbo, AKS + g * kAkStage, Rec::kAkSbo);
      bulk_commit();
    }
    // ---- MMA 1: [A_kk ; A_qk] = [Kp ; Qp] Kn^T   (M=128, N=64, K=128)
    // (kTake) the item three ahead is taken while MMA 1 runs (the atomic's
    // round trip overlaps the wait) and written for the other threads, who
    // read it after this item's last barrier
    int64_t taken = 0;
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        mma_bf16(tmem, sdesc(smem_u32(A1) + s * 2 * kA1Lbo, kA1Lbo, 128),
                 sdesc(smem_u32(B1) + s * 2 * kB1Lbo, kB1Lbo, 128), id, s > 0);
      mma_commit(&bar_mma);
      if (kTake) taken = take_item(p, x);
    }
    // the A_kk tile is rewritten below: the AK copies must have read it
    if (copy_group(tid) >= 0) bulk_wait_read_all();
    ok = bs.all(mbar_wait_t<kPoll>(&bar_mma, 0, p.wait_ns));
    if (kTake && tid == 0) ahead[(nth + 3) & 3] = taken;
    fence_after_sync();
    if (!ok) break;
    if (rescale) {
      // Qp = Qp' 2^s for the record (rows 64-127 of A1, this thread's 4 rows
      // and 8 channels); the bulk copy that reads them comes after a barrier
      const float4 s0 = *reinterpret_cast<const float4*>(sref + c0);
      const float4 s1 = *reinterpret_cast<const float4*>(sref + c0 + 4);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        uint4* u = reinterpret_cast<uint4*>(A1 + kmaj(64 + i0 + r, c0, kA1Lbo));
        const uint4 x = *u;
        *u = make_uint4(pack_bf16(bf16_lo(x.x) * s0.x, bf16_hi(x.x) * s0.y),
                        pack_bf16(bf16_lo(x.y) * s0.z, bf16_hi(x.y) * s0.w),
                        pack_bf16(bf16_lo(x.z) * s1.x, bf16_hi(x.z) * s1.y),
                        pack_bf16(bf16_lo(x.w) * s1.z, bf16_hi(x.w) * s1.w));
      }
    }
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
          *reinterpret_cast<uint4*>(A2 + kmajor_off(i, 8 * jb, 64)) =
              make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                         pack_bf16(a[6], a[7]));
        }
      }
    }
    fence_async_smem();
    fence_before_sync();
    bs.sync();
    // A_qk, staged in A2, to the record
    if (tid == kAqCopy) {
      bulk_s2g(rec + Rec::AQ, A2, 64 * 64 * 2);
      bulk_commit();
    }

    // ---- T = (I + A_kk)^{-1}; Tb = T diag(beta) -> A2 (bf16, R=64)
    tri_inverse_64(AKK, TT, XS, tid == kAqCopy, tid, bs);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int idx = tid + kThreads * t;
      const int i = idx >> 3, jb = idx & 7;  // lanes along a row of T: few bank conflicts
      const float4 t0 = *reinterpret_cast<const float4*>(TT + tsw(i, 8 * jb));
      const float4 t1 = *reinterpret_cast<const float4*>(TT + tsw(i, 8 * jb) + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(beta + 8 * jb);
      const float4 b1 = *reinterpret_cast<const float4*>(beta + 8 * jb + 4);
      st_s16(A2, kmaj(i, 8 * jb, kA2Lbo),
             make_uint4(pack_bf16(t0.x * b0.x, t0.y * b0.y), pack_bf16(t0.z * b0.z, t0.w * b0.w),
                        pack_bf16(t1.x * b1.x, t1.y * b1.y), pack_bf16(t1.z * b1.z, t1.w * b1.w)));
    }
    fence_async_smem();
    fence_before_sync();
    bs.sync();
    fence_after_sync();

    // T is consumed (B1) and the A_kk tile free: the next item's g and k
    // (group A) are staged now
    if (has_next) {
      if (tid == 0) stage_a<kHeadGate, kConv>(sm, &bar_ga, chn, hn, maps);
      bnext = load_b(p, chn, hn, tid);
      if (kHeadGate) gnext = load_gh(p, chn, hn, tid);
      a_fly = true;
    }
    // ---- MMA 2: [W | U~] = Tb [Kp | V]   (M=64, N=256, K=64)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(64, 256, 0, 1);  // B2 is MN-major
#pragma unroll
      for (int s = 0; s < 4; ++s)
        mma_bf16(tmem, sdesc(smem_u32(A2) + s * 2 * kA2Lbo, kA2Lbo, 128),
                 sdesc(smem_u32(B2) + s * 256, 128, kB2Sbo), id, s > 0);
      mma_commit(&bar_mma);
    }
    ok = bs.all(mbar_wait_t<kPoll>(&bar_mma, 1, p.wait_ns));
    fence_after_sync();
    if (!ok) break;
    // MMA 2 has read B2: the next item's q and v (group B) are staged there now
    if (has_next) {
      if (tid == 0) stage_b<kConv>(sm, &bar_gb, chn, hn, maps, p);
      b_fly = true;
    }
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
              st_s16(A1, kmaj(i, c + 8 * u, kA1Lbo),
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
    // the next item's decay logits (gate per head): this item's scan is done
    if (kHeadGate && has_next && tid < 64) gtok[tid] = gnext;
    fence_async_smem();
    fence_before_sync();
    bs.sync();
    fence_after_sync();
    // [W ; Qp] to the record's unpadded layout, one bulk copy per 8-channel
    // group, each from its own thread; their reads are awaited before A1 is
    // rewritten by the next item
    if (copy_group(tid) >= 0) {
      const int g = copy_group(tid);
      bulk_s2g(rec + Rec::AW + g * 128 * 16, A1 + g * kA1Lbo, 128 * 16);
      bulk_commit();
    }
    if (kFused && tid == 0) x.bars->pend = x.bars->cur;
    const int64_t item3 = item_ahead(nth, 3);
    ch = ch_next;
    ch_next = ch_next2;
    ch_next2 = item3 < n_items ? item_chunk<kConv>(p, item3 / H) : ItemChunk{0, 0, 0};
    item = item1;
    ++nth;
  }
  // no staging copy and no MMA is left in flight when the CTA exits (these
  // waits keep the long limit whatever the caller chose for the others)
  if (a_fly) mbar_wait(&bar_ga, sph, kWaitLimitNs);
  if (b_fly) mbar_wait(&bar_gb, sph, kWaitLimitNs);
  if (tid == 0 && !ok) {
    flag(p.status, kFlagTimeout);
    mma_commit(&bar_drain);
    mbar_wait(&bar_drain, 0, kWaitLimitNs);
  }
  bulk_wait_all();  // every thread's own copies
  if constexpr (kFused) {
    // publish the last record (not on the error path: the chains waiting
    // for it give up on their own limit)
    if (copy_group(tid) >= 0) fence_proxy_async_global();
    if (writes_record_rows(tid)) fence_gpu();
    bs.sync();
    if (tid == 0 && ok && x.bars->pend) st_release_u32(x.bars->pend, 1u);
  }
}

// [T][H][D] bf16 rows, box {128 channels, 1 head, `rows` tokens}, zero fill
// outside [0, T) and, for a head of D = 64 channels, in channels 64-127: the
// kernel then runs on the head zero-padded to 128 channels, which leaves
// every product of q^, k^ and v unchanged
bool encode_rows(CUtensorMap* m, const void* base, int H, int64_t T, int D, uint32_t rows = 64) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  const cuuint32_t box[3] = {kD, 1, rows};
  const cuuint32_t elem[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor maps of the call's q, k, v, g (and the convolution's halo
// rows); false if one cannot be encoded
bool make_row_maps(const ChunkParams& p, RowMaps* maps) {
  const bool head = p.gate_per_head != 0, conv = p.conv_width > 0;
  // with a gate per head there are no g rows to stage (the g map is not used)
  const int64_t T = p.total_tokens;
  if (!encode_rows(&maps->g, head ? p.k : p.g, p.H, T, p.dk) || !encode_rows(&maps->q, p.q, p.H, T, p.dk) ||
      !encode_rows(&maps->k, p.k, p.H, T, p.dk) || !encode_rows(&maps->v, p.v, p.H, T, p.dv))
    return false;
  if (conv && (!encode_rows(&maps->qh, p.q, p.H, T, p.dk, kHaloRows) ||
               !encode_rows(&maps->kh, p.k, p.H, T, p.dk, kHaloRows) ||
               !encode_rows(&maps->vh, p.v, p.H, T, p.dv, kHaloRows)))
    return false;
  return true;
}

}  // namespace
}  // namespace tcp
}  // namespace kda
