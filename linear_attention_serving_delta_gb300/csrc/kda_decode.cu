// kda_decode.cu -- one decode step of the KDA recurrence for a batch of rows.
//
// "Kimi K3: The Manos, The Mythos, The Legendos" (bullet on FlashKDA): decode
// costs the same at every position because each step only advances a
// fixed-size state by one token.  Per (row, head) the step is
//
//   S' = Diag(alpha) S                 p = S'^T k^       u = beta (v - p)
//   S  = S' + k^ u^T                   o = scale S^T q^ = scale (S'^T q^ + (q^.k^) u)
//
// (delta rule with a per-channel gate, "From KV Cache to Depth Attention",
// Technical Details).  The work is ~7 dk dv flops per 8 dk dv bytes of state
// traffic, so the kernel is bound by HBM: it reads the fp32 state once into
// registers with 16-byte coalesced loads (a warp covers whole 512-byte rows
// for dv = 128), reduces S'^T k^ and S'^T q^ over the key channels in
// registers and through shared memory, and writes the state back once.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

// ---------------------------------------------------------- layer steps
// The short convolution of one input channel for one decode token ("Kimi K3:
// The Manos, The Mythos, The Legendos", bullet on the stability details;
// formula in include/kda.h): tap 0 on the token's own input x, tap j on the
// input j tokens back, which is row W - 1 - j of the slot's window (zeros
// without one); SiLU if asked; rounded to the input dtype.  `prev(m)` reads
// window row m.
template <typename TIn, typename Prev>
__device__ __forceinline__ float conv_token(const kda_layer_args& l, int t, float x, int H, int h, int c, int d,
                                            Prev prev) {
  const int W = l.conv_width;
  const float* w = l.conv_w[t];
  float acc = w[(int64_t)h * d + c] * x;
  for (int j = 1; j < W; ++j) acc += w[((int64_t)j * H + h) * d + c] * prev(W - 1 - j);
  if (l.conv_silu) acc = silu_of(acc);
  return round_in<TIn>(acc);
}
// Row m of the window of tensor t in global memory (slot's rows), 0 without one
template <typename TIn>
__device__ __forceinline__ float window_at(const kda_layer_args& l, int t, int slot, int m, int H, int h, int c,
                                           int d) {
  const TIn* win = static_cast<const TIn*>(l.conv_in[t]);
  return win ? ld_in(win, (((int64_t)slot * (l.conv_width - 1) + m) * H + h) * d + c) : 0.f;
}
// The window after the token: rows shift down by one (row m <- row m + 1) and
// the last row takes the raw input x.  Reads precede writes per element, so
// conv_out may be conv_in.
template <typename TIn, typename Prev>
__device__ __forceinline__ void window_push(const kda_layer_args& l, int t, float x, int slot, int H, int h,
                                            int c, int d, Prev prev) {
  const int W = l.conv_width;
  TIn* out = static_cast<TIn*>(l.conv_out[t]);
  if (W <= 1 || !out) return;
  const int64_t base = (int64_t)slot * (W - 1);
  for (int m = 0; m + 1 < W - 1; ++m) st_out(out, ((base + m) * H + h) * d + c, prev(m + 1));
  st_out(out, ((base + W - 2) * H + h) * d + c, x);
}
// the output gate's factor for o element `e` of row `row`, head h (1 without a gate)
template <typename TIn>
__device__ __forceinline__ float gate_at(const kda_layer_args& l, int64_t row, int H, int h, int64_t e) {
  if (!l.out_gate) return 1.f;
  const TIn* r = static_cast<const TIn*>(l.out_gate);
  return out_gate_of(ld_in(r, l.out_gate_per_head ? row * H + h : e));
}

template <typename TIn, int DK, int DV>
struct DecodeShape {
  static constexpr int QPR = DV / 4;                           // float4 quads per row
  static constexpr int NT = (QPR * DK < 256) ? QPR * DK : 256; // threads
  static constexpr int NRG = NT / QPR;                         // row groups
  static constexpr int RPT = DK / NRG;                         // rows per thread
  static_assert(DK % NRG == 0, "row groups tile the key channels");
};

// One CTA per (row, head, slice of DVS value columns): the reductions run
// over key channels for each value column, so the columns split freely.
// Heads up to 128 x 128 take one slice (DVS = DV); wider ones slices of 64,
// which keep a thread's share of the state in registers.
template <int DK, int DV>
struct DecodeSlice {
  static constexpr int DVS = DK * DV > 128 * 128 ? 64 : DV;
};

template <typename TIn, int DK, int DV, int DVS>
__global__ void __launch_bounds__(DecodeShape<TIn, DK, DVS>::NT)
decode_step(kda_decode_args a, const kda_layer_args l) {
  using Sh = DecodeShape<TIn, DK, DVS>;
  constexpr int QPR = Sh::QPR, NT = Sh::NT, NRG = Sh::NRG, RPT = Sh::RPT;
  // arrays read through float4 are 16-byte aligned explicitly
  __shared__ __align__(16) float qn[DK];
  __shared__ __align__(16) float kn[DK];
  __shared__ __align__(16) float al[DK];
  __shared__ __align__(16) float vv[DVS];
  __shared__ __align__(16) float red_p[NRG][DVS];
  __shared__ __align__(16) float red_o[NRG][DVS];
  __shared__ float sc[2];  // beta, q^.k^

  const int row = blockIdx.x, h = blockIdx.y, H = a.num_heads, n0 = blockIdx.z * DVS;
  const int slot = a.state_slots ? a.state_slots[row] : row;
  if (slot < 0 || slot >= a.num_slots) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cq = tid % QPR, rg = tid / QPR;
  float* S = a.state + ((size_t)slot * H + h) * DK * DV;

  // stream this thread's rows of the state into registers first
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i)
    s[i] = reinterpret_cast<const float4*>(S + (size_t)(rg + i * NRG) * DV + n0)[cq];

  // token preparation (one warp): q^, k^, alpha, beta, q^.k^
  if (warp == 0) {
    const TIn* q = static_cast<const TIn*>(a.q);
    const TIn* k = static_cast<const TIn*>(a.k);
    const TIn* g = static_cast<const TIn*>(a.g);
    const TIn* v = static_cast<const TIn*>(a.v);
    const int64_t base_k = ((int64_t)row * H + h) * DK;
    const int64_t base_v = ((int64_t)row * H + h) * DV;
    float sq = 0.f, sk = 0.f;
    for (int c = lane; c < DK; c += 32) {
      float xq = ld_in(q, base_k + c), xk = ld_in(k, base_k + c);
      if (l.conv_width > 0) {
        auto pq = [&](int m) { return window_at<TIn>(l, 0, slot, m, H, h, c, DK); };
        auto pk = [&](int m) { return window_at<TIn>(l, 1, slot, m, H, h, c, DK); };
        const float rq = xq, rk = xk;
        xq = conv_token<TIn>(l, 0, rq, H, h, c, DK, pq);
        xk = conv_token<TIn>(l, 1, rk, H, h, c, DK, pk);
        window_push<TIn>(l, 0, rq, slot, H, h, c, DK, pq);
        window_push<TIn>(l, 1, rk, slot, H, h, c, DK, pk);
      }
      qn[c] = xq;
      kn[c] = xk;
      al[c] = expf(log_alpha_of(ld_in(g, a.gate_per_head ? (int64_t)row * H + h : base_k + c)));
      sq += xq * xq;
      sk += xk * xk;
    }
    for (int cs = lane; cs < DVS; cs += 32) {
      const int c = n0 + cs;
      float xv = ld_in(v, base_v + c);
      if (l.conv_width > 0) {
        auto pv = [&](int m) { return window_at<TIn>(l, 2, slot, m, H, h, c, DV); };
        const float rv = xv;
        xv = conv_token<TIn>(l, 2, rv, H, h, c, DV, pv);
        window_push<TIn>(l, 2, rv, slot, H, h, c, DV, pv);
      }
      vv[cs] = xv;
    }
    const float iq = inv_norm_of(warp_sum(sq)), ik = inv_norm_of(warp_sum(sk));
    float qk = 0.f;
    for (int c = lane; c < DK; c += 32) {
      qn[c] *= iq;
      kn[c] *= ik;
      qk += qn[c] * kn[c];
    }
    qk = warp_sum(qk);
    if (lane == 0) {
      sc[0] = beta_of(ld_in(static_cast<const TIn*>(a.b), (int64_t)row * H + h));
      sc[1] = qk;
    }
  }
  __syncthreads();

  // retention and the two reductions over key channels
  float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), po = pp;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * NRG;
    const float a_r = al[r], k_r = kn[r], q_r = qn[r];
    s[i].x *= a_r; s[i].y *= a_r; s[i].z *= a_r; s[i].w *= a_r;
    pp.x += k_r * s[i].x; pp.y += k_r * s[i].y; pp.z += k_r * s[i].z; pp.w += k_r * s[i].w;
    po.x += q_r * s[i].x; po.y += q_r * s[i].y; po.z += q_r * s[i].z; po.w += q_r * s[i].w;
  }
  // row groups that share a warp (dv < 128) combine with shuffles first
  constexpr int RGW = 32 / QPR;  // row groups per warp
#pragma unroll
  for (int off = QPR; off < 32 && RGW > 1; off <<= 1) {
    pp.x += __shfl_xor_sync(0xffffffffu, pp.x, off);
    pp.y += __shfl_xor_sync(0xffffffffu, pp.y, off);
    pp.z += __shfl_xor_sync(0xffffffffu, pp.z, off);
    pp.w += __shfl_xor_sync(0xffffffffu, pp.w, off);
    po.x += __shfl_xor_sync(0xffffffffu, po.x, off);
    po.y += __shfl_xor_sync(0xffffffffu, po.y, off);
    po.z += __shfl_xor_sync(0xffffffffu, po.z, off);
    po.w += __shfl_xor_sync(0xffffffffu, po.w, off);
  }
  constexpr int NW = NT / 32 > 0 ? NT / 32 : 1;
  const bool writer = (RGW > 1) ? (lane < QPR) : true;
  const int slotw = (RGW > 1) ? warp : rg;
  if (writer) {
    *reinterpret_cast<float4*>(&red_p[slotw][4 * cq]) = pp;
    *reinterpret_cast<float4*>(&red_o[slotw][4 * cq]) = po;
  }
  __syncthreads();
  const int nred = (RGW > 1) ? NW : NRG;
  float4 p = make_float4(0.f, 0.f, 0.f, 0.f), oq = p;
  for (int w = 0; w < nred; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(&red_p[w][4 * cq]);
    const float4 y = *reinterpret_cast<const float4*>(&red_o[w][4 * cq]);
    p.x += x.x; p.y += x.y; p.z += x.z; p.w += x.w;
    oq.x += y.x; oq.y += y.y; oq.z += y.z; oq.w += y.w;
  }
  const float beta = sc[0];
  const float4 vq = *reinterpret_cast<const float4*>(&vv[4 * cq]);
  const float4 u = make_float4(beta * (vq.x - p.x), beta * (vq.y - p.y), beta * (vq.z - p.z),
                               beta * (vq.w - p.w));
  // rank-1 write of the delta, state written back once
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * NRG;
    const float k_r = kn[r];
    float4 x = s[i];
    x.x += k_r * u.x; x.y += k_r * u.y; x.z += k_r * u.z; x.w += k_r * u.w;
    reinterpret_cast<float4*>(S + (size_t)r * DV + n0)[cq] = x;
  }
  if (rg == 0) {
    const float qk = sc[1], scl = a.scale;
    TIn* o = static_cast<TIn*>(a.o);
    const int64_t ob = ((int64_t)row * H + h) * DV + n0 + 4 * cq;
    st_out(o, ob + 0, scl * (oq.x + qk * u.x) * gate_at<TIn>(l, row, H, h, ob + 0));
    st_out(o, ob + 1, scl * (oq.y + qk * u.y) * gate_at<TIn>(l, row, H, h, ob + 1));
    st_out(o, ob + 2, scl * (oq.z + qk * u.z) * gate_at<TIn>(l, row, H, h, ob + 2));
    st_out(o, ob + 3, scl * (oq.w + qk * u.w) * gate_at<TIn>(l, row, H, h, ob + 3));
  }
}

// ------------------------------------------------- dk, dv in {64, 128, 256}
// Persistent variant: one CTA per SM walks (row, head, column slice) items.
// A ring of shared-memory slots is filled by copies (TMA engine) of each
// item's state plus its q, k, g, v rows, a few items ahead (3 slots of 64 KB
// states, up to 8 for smaller states, so that about 200 KB stay in flight
// per SM).  A head of at most 64 KB of state (up to 128 x 128, or 256 x 64,
// 64 x 256) is one item, its state one contiguous 1-D bulk copy; a larger
// head (dk or dv = 256) is cut into slices of DVS value columns that hold
// 64 KB each (256 x 64, 128 x 128), moved in and out by 2-D tensor-map
// copies of the strided slice: the reductions over key channels are per
// value column, so the slices of a head are independent (each reads the
// head's whole q, k and g rows and its own columns of v).
// Warps 0-7 compute; warp 8 is the producer: once the compute warps have
// written an item's updated state into its slot, it sends the state back to
// HBM with one 64 KB bulk copy, waits for that copy to read the slot and
// refills it with the item kStages further on.  No compute warp waits on a
// copy.
//
// The compute warps need no token-preparation phase: with raw q, k,
// p = S'^T k^ = ik (S'^T k) and S'^T q^ = iq (S'^T q) (ik, iq the inverse
// norms), so each warp reads q, k and g of its own DK / 8 key channels
// straight from the slot, and the norms' partial sums travel with the
// reduction partials through the one barrier of the item.
constexpr int kRingThreads = 256;            // compute warps 0-7
constexpr int kRingAllThreads = kRingThreads + 32;  // + the producer warp
constexpr int kComputeBarrier = 1;           // named barrier of warps 0-7

// A slot: the state, the q, k, g, v rows and, with the short convolution,
// up to KDA_CONV_MAX - 1 window rows of each of q, k, v.  Warp w owns key
// rows w + 8 i (i < RPW), lane l value columns CPL l .. CPL l + CPL - 1.
constexpr int kWinRows = KDA_CONV_MAX - 1;
// Value columns per item of a dk x dv head: at most 128 (a lane's 2 or 4
// columns of a row are one 8- or 16-byte access) and at most 64 KB of state
template <int DK, int DV>
struct RingSlice {
  static constexpr int CAP = 128 * 128 / DK < 128 ? 128 * 128 / DK : 128;
  static constexpr int DVS = DV < CAP ? DV : CAP;
  static constexpr int NS = DV / DVS;  // slices per head
};
// G heads per item: consecutive heads of one row are adjacent in the pool
// and in q, k, g, v, so a slot of G small heads (G x 16 or 32 KB) is filled
// by the same few copies as one large head, and an item's fixed costs are
// shared by G heads.  8 / G compute warps per head.
template <typename TIn, bool kConv, int DK, int DV, int G = 1>
struct Ring {
  static constexpr int DVS = RingSlice<DK, DV>::DVS, NS = RingSlice<DK, DV>::NS;
  static_assert((DK == 64 || DK == 128 || DK == 256) && (DVS == 64 || DVS == 128) && DK * DVS <= 128 * 128,
                "ring head sizes");
  static_assert(G == 1 || (NS == 1 && !kConv && G * DK * DVS <= 128 * 128 && (G == 2 || G == 4)),
                "several heads per item: unsliced heads, no convolution, at most 64 KB of state");
  static constexpr int WH = 8 / G;                   // compute warps per head
  static constexpr int RPW = DK / WH, CPL = DVS / 32;
  static constexpr uint32_t STATE = G * DK * DVS * 4;
  static constexpr uint32_t RK = G * DK * sizeof(TIn), RV = G * DVS * sizeof(TIn);  // q / k / g rows, v
  static constexpr uint32_t QO = STATE, KO = QO + RK, GO = KO + RK, VO = GO + RK;
  static constexpr uint32_t RW = RK > RV ? RK : RV;
  static constexpr uint32_t WIN = VO + RV;  // window row m of tensor t at WIN + (3 m + t) RW
  // (128-byte multiple: the tensor-map copy of the next slot's state lands on
  // a 128-byte boundary)
  static constexpr uint32_t STAGE = (WIN + (kConv ? 3 * kWinRows * RW : 0) + 127) / 128 * 128;
  // 64 x 64 states (16 KB) run two CTAs per SM: an item's fixed costs (two
  // barriers, the reductions) then overlap with the other CTA's
  static constexpr int CTAS = STATE <= 16384 ? 2 : 1;
  static constexpr uint32_t BUDGET = CTAS == 2 ? 96000 : 200000;
  static constexpr int STAGES = BUDGET / STAGE < 3 ? 3 : (BUDGET / STAGE > 8 ? 8 : BUDGET / STAGE);
  static constexpr uint32_t BYTES = STAGES * STAGE;
};

// CPL consecutive floats (one 8- or 16-byte access)
template <int CPL>
__device__ __forceinline__ void ld_cols(const float* p, float* x) {
  if constexpr (CPL == 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    const float2 v = *reinterpret_cast<const float2*>(p);
    x[0] = v.x; x[1] = v.y;
  }
}
template <int CPL>
__device__ __forceinline__ void st_cols(float* p, const float* x) {
  if constexpr (CPL == 4)
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// barrier.red.and over the `n` threads of named barrier `id`
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, p;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// The state of a slice item as a box of the pool viewed as [slots H DK][DV]
// fp32 rows: DVS columns x DK rows at (column z DVS, row (slot H + h) DK)
__device__ __forceinline__ void tma_state_load(uint8_t* dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(tc::smem_u32(dst)),
      "l"(m), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_state_store(const CUtensorMap* m, int x, int y, const uint8_t* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(m), "r"(x),
               "r"(y), "r"(tc::smem_u32(src))
               : "memory");
}

// An item: (row, first head h, slice z) with the slices of one head
// adjacent; with G heads per item (NS = 1), heads h .. h + G - 1
struct RingItem {
  int row, h, z;
};
template <int NS, int G = 1>
__device__ __forceinline__ RingItem ring_item(int64_t item, int H) {
  if (G > 1) {
    const int hg = H / G;
    return RingItem{(int)(item / hg), (int)(item % hg) * G, 0};
  }
  const int64_t rh = item / NS;
  return RingItem{(int)(rh / H), (int)(rh % H), (int)(item % NS)};
}
// index of (row, head h + gi) in a [B, H] tensor (b, g with a gate per head)
template <int NS, int G = 1>
__device__ __forceinline__ int64_t ring_rowhead(int64_t item, int gi) {
  return (item / NS) * G + gi;
}

template <typename TIn, bool kConv, int DK, int DV, int G>
__device__ __forceinline__ void ring_issue(const kda_decode_args& a, const kda_layer_args& l, uint8_t* stage,
                                           uint64_t* bar, int32_t* valid_flag, int64_t item,
                                           const CUtensorMap* smap) {
  using R = Ring<TIn, kConv, DK, DV, G>;
  const int H = a.num_heads;
  const RingItem it = ring_item<R::NS, G>(item, H);
  const int row = it.row, h = it.h;
  const int slot = a.state_slots ? a.state_slots[row] : row;
  const bool valid = slot >= 0 && slot < a.num_slots;
  *valid_flag = valid ? 1 : 0;
  if (!valid) {
    mbar_arrive(bar);
    return;
  }
  // (with a gate per head there is no g row: the compute warps read its one value)
  uint32_t bytes = R::STATE + (a.gate_per_head ? 2 : 3) * R::RK + R::RV;
  const int nw = kConv ? l.conv_width - 1 : 0;  // window rows per tensor
  if (kConv)
    for (int t = 0; t < 3; ++t)
      if (l.conv_in[t]) bytes += nw * (t == 2 ? R::RV : R::RK);
  tc::mbar_arrive_expect_tx(bar, bytes);
  const int64_t ek = ((int64_t)row * H + h) * DK, ev = ((int64_t)row * H + h) * DV + it.z * R::DVS;
  if (R::NS > 1)
    tma_state_load(stage, smap, it.z * R::DVS, (slot * H + h) * DK, bar);
  else
    tc::bulk_g2s(stage, a.state + ((size_t)slot * H + h) * DK * DV, R::STATE, bar);
  tc::bulk_g2s(stage + R::QO, static_cast<const TIn*>(a.q) + ek, R::RK, bar);
  tc::bulk_g2s(stage + R::KO, static_cast<const TIn*>(a.k) + ek, R::RK, bar);
  if (!a.gate_per_head) tc::bulk_g2s(stage + R::GO, static_cast<const TIn*>(a.g) + ek, R::RK, bar);
  tc::bulk_g2s(stage + R::VO, static_cast<const TIn*>(a.v) + ev, R::RV, bar);
  if (kConv)
    for (int t = 0; t < 3; ++t)
      if (l.conv_in[t]) {
        const int d = t == 2 ? DV : DK;
        for (int m = 0; m < nw; ++m)
          tc::bulk_g2s(stage + R::WIN + (3 * m + t) * R::RW,
                       static_cast<const TIn*>(l.conv_in[t]) + (((int64_t)slot * nw + m) * H + h) * d,
                       d * (uint32_t)sizeof(TIn), bar);
      }
}

// kPoll: the instantiation for wait limits under kPollLimitNs (the give-up
// test).  kConv: the short convolution (window rows in the slot).
// smap: the pool as [slots H DK][DV] fp32 rows with a box of DVS columns x
// DK rows (used when a head is cut into slices)
template <typename TIn, bool kPoll, bool kConv, int DK, int DV, int G>
__global__ void __launch_bounds__(kRingAllThreads, (G * DK * DV <= 64 * 64) ? 2 : 1)
decode_ring(kda_decode_args a, int64_t n_items, const kda_layer_args l, const __grid_constant__ CUtensorMap smap) {
  using R = Ring<TIn, kConv, DK, DV, G>;
  constexpr int kStages = R::STAGES, RPW = R::RPW, CPL = R::CPL, DVS = R::DVS, NS = R::NS, WH = R::WH;
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[kStages];  // slot loaded
  __shared__ __align__(8) uint64_t done[kStages];  // slot's state updated by warps 0-7
  __shared__ int32_t valid_flag[kStages];
  __shared__ __align__(16) float red_p[2][8][DVS];
  __shared__ __align__(16) float red_o[2][8][DVS];
  __shared__ __align__(16) float part[2][8][4];    // per warp: sum q^2, sum k^2, sum q k
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.num_heads;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t n_local = first < n_items ? (n_items - first + stride - 1) / stride : 0;

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      tc::mbar_init(&full[st], 1);
      tc::mbar_init(&done[st], kRingThreads);
    }
    tc::mbar_init_fence();
  }
  // (launched as the programmatic dependent of the kernel before it, the
  // previous decode step on the same pool as a rule) nothing it wrote is
  // read before this point; the next step may be launched now (its CTAs
  // take the SMs this one leaves and wait there likewise)
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();

  const uint64_t lim = a.wait_limit_ns > 0 ? (uint64_t)a.wait_limit_ns : tc::kWaitLimitNs;
  if (warp == 8) {
    // ---- producer
    if (lane == 0) {
      int64_t issued = 0;  // items whose slot copies were issued
      for (; issued < kStages && issued < n_local; ++issued)
        ring_issue<TIn, kConv, DK, DV, G>(a, l, sm + issued * R::STAGE, &full[issued], &valid_flag[issued],
                                          first + issued * stride, &smap);
      for (int64_t k = 0; k < n_local; ++k) {
        const int st = (int)(k % kStages);
        uint8_t* stage = sm + st * R::STAGE;
        if (!tc::mbar_wait_t<kPoll>(&done[st], (uint32_t)((k / kStages) & 1), lim)) {
          // the compute warps gave up: let the slot copies still in flight
          // land (long limit) before the shared memory is given back
          if (a.status) atomicOr(a.status, kFlagTimeout);
          for (int64_t j = k; j < issued; ++j)
            tc::mbar_wait(&full[j % kStages], (uint32_t)((j / kStages) & 1), tc::kWaitLimitNs);
          break;
        }
        const int64_t item = first + k * stride;
        if (valid_flag[st]) {
          const RingItem it = ring_item<NS, G>(item, H);
          const int slot = a.state_slots ? a.state_slots[it.row] : it.row;
          if (NS > 1)
            tma_state_store(&smap, it.z * DVS, (slot * H + it.h) * DK, stage);
          else
            tc::bulk_s2g(a.state + ((size_t)slot * H + it.h) * DK * DV, stage, R::STATE);
          tc::bulk_commit();
          tc::bulk_wait_read_all();
        }
        if (k + kStages < n_local) {
          ring_issue<TIn, kConv, DK, DV, G>(a, l, stage, &full[st], &valid_flag[st], item + kStages * stride,
                                            &smap);
          issued = k + kStages + 1;
        }
      }
      tc::bulk_wait_all();
    }
    return;
  }

  // ---- compute warps 0-7: warp w works on head gi = w / WH of the item and
  // owns its key channels (rows) lw + WH i, i < RPW (lw = w % WH)
  const int gi = warp / WH, lw = warp % WH;
  const TIn* gb = static_cast<const TIn*>(a.b);
  // b [B, H]: one per (row, head)
  float b_next = n_local > 0 ? ld_in(gb, ring_rowhead<NS, G>(first, gi)) : 0.f;
  for (int64_t k = 0; k < n_local; ++k) {
    const int st = (int)(k % kStages);
    uint8_t* stage = sm + st * R::STAGE;
    const int64_t item = first + k * stride;
    const int buf = (int)(k & 1);
    bool ok = tc::mbar_wait_t<kPoll>(&full[st], (uint32_t)((k / kStages) & 1), lim);
    const bool valid = valid_flag[st] != 0;
    const float b_cur = b_next;
    if (k + 1 < n_local) b_next = ld_in(gb, ring_rowhead<NS, G>(item + stride, gi));
    if (!valid) {  // uniform: nothing to compute, the slot is handed back
      mbar_arrive(&done[st]);
      if (!bar_and(kComputeBarrier, kRingThreads, ok)) {
        if (tid == 0 && a.status) atomicOr(a.status, kFlagTimeout);
        break;
      }
      continue;
    }
    // this warp's head's rows of q, k, g, v in the slot
    const TIn* rq = reinterpret_cast<const TIn*>(stage + R::QO) + gi * DK;
    const TIn* rk = reinterpret_cast<const TIn*>(stage + R::KO) + gi * DK;
    const TIn* rg = reinterpret_cast<const TIn*>(stage + R::GO) + gi * DK;
    const TIn* rv = reinterpret_cast<const TIn*>(stage + R::VO) + gi * DVS;
    // this warp's RPW rows: lane i < RPW holds raw q, k and alpha of row lw + WH i
    float xq = 0.f, xk = 0.f, xa = 0.f;
    // with the convolution: window row m of tensor t in the slot (0 without one)
    auto wrow = [&](int t, int m, int c) {
      return l.conv_in[t] ? ld_in(reinterpret_cast<const TIn*>(stage + R::WIN + (3 * m + t) * R::RW), c) : 0.f;
    };
    const RingItem it = ring_item<NS, G>(item, H);
    int slot = 0;
    if (kConv) slot = a.state_slots ? a.state_slots[it.row] : it.row;
    const int hh = it.h;
    if (lane < RPW) {
      const int r = lw + WH * lane;
      xq = ld_in(rq, r);
      xk = ld_in(rk, r);
      xa = expf(log_alpha_of(a.gate_per_head ? ld_in(static_cast<const TIn*>(a.g), ring_rowhead<NS, G>(item, gi))
                                             : ld_in(rg, r)));
      if (kConv) {
        auto pq = [&](int m) { return wrow(0, m, r); };
        auto pk = [&](int m) { return wrow(1, m, r); };
        window_push<TIn>(l, 0, xq, slot, H, hh, r, DK, pq);
        window_push<TIn>(l, 1, xk, slot, H, hh, r, DK, pk);
        xq = conv_token<TIn>(l, 0, xq, H, hh, r, DK, pq);
        xk = conv_token<TIn>(l, 1, xk, H, hh, r, DK, pk);
      }
    }
    {
      const float sq = warp_sum(xq * xq), sk = warp_sum(xk * xk), sqk = warp_sum(xq * xk);
      if (lane == 0) *reinterpret_cast<float4*>(&part[buf][warp][0]) = make_float4(sq, sk, sqk, 0.f);
    }
    // retention and the two reductions over this warp's rows (raw q, k)
    const float* S = reinterpret_cast<const float*>(stage) + gi * DK * DVS;
    float s[RPW][CPL], pp[CPL], po[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) pp[j] = po[j] = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int r = lw + WH * i;
      ld_cols<CPL>(S + r * DVS + CPL * lane, s[i]);
      const float a_r = __shfl_sync(0xffffffffu, xa, i), k_r = __shfl_sync(0xffffffffu, xk, i),
                  q_r = __shfl_sync(0xffffffffu, xq, i);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        s[i][j] *= a_r;
        pp[j] += k_r * s[i][j];
        po[j] += q_r * s[i][j];
      }
    }
    st_cols<CPL>(&red_p[buf][warp][CPL * lane], pp);
    st_cols<CPL>(&red_o[buf][warp][CPL * lane], po);
    if (!bar_and(kComputeBarrier, kRingThreads, ok)) {
      if (tid == 0 && a.status) atomicOr(a.status, kFlagTimeout);
      break;
    }
    // the partial sums of this head's warps
    float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
    for (int w = gi * WH; w < gi * WH + WH; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(&part[buf][w][0]);
      sq += x.x; sk += x.y; sqk += x.z;
    }
    const float iq = inv_norm_of(sq), ik = inv_norm_of(sk), qk = sqk * iq * ik;
    float p[CPL], oq[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) p[j] = oq[j] = 0.f;
#pragma unroll
    for (int w = gi * WH; w < gi * WH + WH; ++w) {
      float x[CPL], y[CPL];
      ld_cols<CPL>(&red_p[buf][w][CPL * lane], x);
      ld_cols<CPL>(&red_o[buf][w][CPL * lane], y);
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        p[j] += x[j];
        oq[j] += y[j];
      }
    }
    const float beta = beta_of(b_cur);
    float u[CPL];
#pragma unroll
    for (int t = 0; t < CPL; ++t) {
      const int c = CPL * lane + t;
      float vx = ld_in(rv, c);
      if (kConv) {
        auto pv = [&](int m) { return wrow(2, m, c); };
        if (warp == 0) window_push<TIn>(l, 2, vx, slot, H, hh, c, DV, pv);
        vx = conv_token<TIn>(l, 2, vx, H, hh, c, DV, pv);
      }
      u[t] = beta * (vx - ik * p[t]);
    }
    // the updated state into the slot (each thread its own rows), then the
    // producer sends it back
    float* Ss = reinterpret_cast<float*>(stage) + gi * DK * DVS;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int r = lw + WH * i;
      const float k_r = ik * __shfl_sync(0xffffffffu, xk, i);
#pragma unroll
      for (int j = 0; j < CPL; ++j) s[i][j] += k_r * u[j];
      st_cols<CPL>(Ss + r * DVS + CPL * lane, s[i]);
    }
    tc::fence_async_smem();
    mbar_arrive(&done[st]);
    if (lw == 0) {  // one warp per head writes its o
      const float scl = a.scale;
      const int row = it.row, h = it.h + gi;
      TIn* o = static_cast<TIn*>(a.o);
      const int64_t ob = ((int64_t)row * H + h) * DV + it.z * DVS + CPL * lane;
#pragma unroll
      for (int t = 0; t < CPL; ++t)
        st_out(o, ob + t, scl * (iq * oq[t] + qk * u[t]) * gate_at<TIn>(l, row, H, h, ob + t));
    }
  }
}

// The state pool [slots, H, DK, DV] fp32 as rows of DV columns, box DVS x DK
// (a slice of one head), for the ring's slice copies
template <int DK, int DV>
bool encode_state_map(CUtensorMap* m, const kda_decode_args& a) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)DV, (cuuint64_t)a.num_slots * a.num_heads * DK};
  const cuuint64_t strides[1] = {(cuuint64_t)DV * 4};
  const cuuint32_t box[2] = {(cuuint32_t)RingSlice<DK, DV>::DVS, (cuuint32_t)DK};
  const cuuint32_t elem[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.state, dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename TIn, bool kConv, int DK, int DV, int G = 1>
cudaError_t launch_ring(const kda_decode_args& a, const kda_layer_args& l, cudaStream_t stream) {
  using R = Ring<TIn, kConv, DK, DV, G>;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool poll = a.wait_limit_ns > 0 && (uint64_t)a.wait_limit_ns < tc::kPollLimitNs;
  auto kernel = poll ? decode_ring<TIn, true, kConv, DK, DV, G> : decode_ring<TIn, false, kConv, DK, DV, G>;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)R::BYTES);
  if (e != cudaSuccess) return e;
  CUtensorMap smap{};
  if (R::NS > 1 && !encode_state_map<DK, DV>(&smap, a)) return cudaErrorInvalidValue;
  const int64_t n_items = (int64_t)a.batch * a.num_heads * R::NS / G, slots = (int64_t)sms * R::CTAS;
  const int64_t grid = n_items < slots ? n_items : slots;
  return launch_maybe_dependent(true, kernel, dim3((unsigned)grid), dim3(kRingAllThreads), (size_t)R::BYTES,
                                stream, a, n_items, l, smap);
}

template <typename TIn, int DK, int DV>
cudaError_t launch_t(const kda_decode_args& a, const kda_layer_args& l, cudaStream_t stream) {
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  // the bulk copies of the ring need 16-byte aligned sources; with the
  // convolution the ring takes bf16 only (fp32 window rows overflow its
  // shared memory)
  const bool conv = l.conv_width > 0;
  constexpr bool kRingShape = (DK == 64 || DK == 128 || DK == 256) && (DV == 64 || DV == 128 || DV == 256);
  if constexpr (kRingShape) {
    // heads cut into slices: the tensor-map rows (slot H + h) DK must fit its
    // int32 coordinates, and the slices would share a q/k window (the
    // convolution is refused for these heads anyway)
    constexpr int NS = RingSlice<DK, DV>::NS;
    const bool rows_fit = NS == 1 || (int64_t)a.num_slots * a.num_heads * DK < ((int64_t)1 << 31);
    if (rows_fit && al16(a.q) && al16(a.k) && (a.gate_per_head || al16(a.g)) && al16(a.v) && al16(a.state) &&
        (!conv || (NS == 1 && DK <= 128 && sizeof(TIn) == 2 && al16(l.conv_in[0]) && al16(l.conv_in[1]) &&
                   al16(l.conv_in[2])))) {
      if constexpr (sizeof(TIn) == 2 && NS == 1 && DK <= 128)
        if (conv) return launch_ring<TIn, true, DK, DV>(a, l, stream);
      // small heads: several per item (up to 64 KB of state), when the head
      // count divides into groups of that size
      if constexpr (NS == 1 && 4 * DK * DV <= 128 * 128)
        if (a.num_heads % 4 == 0) return launch_ring<TIn, false, DK, DV, 4>(a, l, stream);
      if constexpr (NS == 1 && 2 * DK * DV <= 128 * 128)
        if (a.num_heads % 2 == 0) return launch_ring<TIn, false, DK, DV, 2>(a, l, stream);
      return launch_ring<TIn, false, DK, DV>(a, l, stream);
    }
  }
  constexpr int DVS = DecodeSlice<DK, DV>::DVS;
  dim3 grid((unsigned)a.batch, (unsigned)a.num_heads, (unsigned)(DV / DVS));
  decode_step<TIn, DK, DV, DVS><<<grid, DecodeShape<TIn, DK, DVS>::NT, 0, stream>>>(a, l);
  return cudaGetLastError();
}

template <typename TIn, int DK>
cudaError_t launch_dv(const kda_decode_args& a, const kda_layer_args& l, cudaStream_t stream) {
  switch (a.dv) {
    case 16: return launch_t<TIn, DK, 16>(a, l, stream);
    case 32: return launch_t<TIn, DK, 32>(a, l, stream);
    case 64: return launch_t<TIn, DK, 64>(a, l, stream);
    case 128: return launch_t<TIn, DK, 128>(a, l, stream);
    case 256: return launch_t<TIn, DK, 256>(a, l, stream);
  }
  return cudaErrorInvalidValue;
}

template <typename TIn>
cudaError_t launch_dk(const kda_decode_args& a, const kda_layer_args& l, cudaStream_t stream) {
  switch (a.dk) {
    case 16: return launch_dv<TIn, 16>(a, l, stream);
    case 32: return launch_dv<TIn, 32>(a, l, stream);
    case 64: return launch_dv<TIn, 64>(a, l, stream);
    case 128: return launch_dv<TIn, 128>(a, l, stream);
    case 256: return launch_dv<TIn, 256>(a, l, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const kda_decode_args& a, cudaStream_t stream) {
  if (a.batch == 0) return cudaSuccess;
  kda_layer_args l{};  // by value: the kernels cannot read the caller's host struct
  if (a.layer) l = *a.layer;
  if (l.conv_width == 0)
    for (int t = 0; t < 3; ++t) l.conv_in[t] = l.conv_out[t] = nullptr;
  return a.in_dtype == KDA_BF16 ? launch_dk<__nv_bfloat16>(a, l, stream) : launch_dk<float>(a, l, stream);
}

}  // namespace kda
