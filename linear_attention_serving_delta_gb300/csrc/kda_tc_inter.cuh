// kda_tc_inter.cuh -- the inter-chunk step of the tensor-core prefill (K3)
// as a device function over one chain CTA, for the inter-chunk kernel
// (kda_tc_inter.cu) and the chain CTAs of the fused kernel (kda_tc_fused.cu).
//
// One CTA of 256 threads per (sequence, head, 32-column slice of S), walking
// the sequence's chunks in order.  The state slice lives in TMEM as fp32
// accumulators (lane = key channel); a bf16 copy of it in shared memory is
// the MMA operand.  Every MMA runs at N=64: the bf16 operand of a 32-column
// fp32 block is its hi half next to its lo half (x = hi + lo to about
// 2^-16), so one instruction multiplies both.  A tcgen05.mma costs about the
// same for any N <= 64, so this doubles the precision of the state and U
// operands for free.  Each thread keeps its 16 state values in fp32
// registers; MMA 2 writes the chunk's increment into two fresh accumulators
// [Da | Db] (the hi and the lo products), and the write-back forms
// S_{j+1} = Gamma_L(j) S_j + Da + Db.
//
// Two warps share each TMEM lane quarter (warps w and w+4), each taking 16 of
// the 32 columns.  Step j of the walk, with S = S_j (the state entering
// chunk j), the operand holding S_j and TMEM holding Gamma_L(j) S_j:
//   thread 0:      MMA 1 (M=128, N=64, K=128): [W ; Qp] [S_hi | S_lo] -> D1[j % 3]
//   warps 2,3,6,7: the output rows of chunk j-2 (its MMA 3 is done), copies;
//                  thread 64 then issues MMA 3 of chunk j-1 (M=128, N=64,
//                  K=64): D1[(j-1) % 3][64..127] += A_qk [U_hi | U_lo]
//   warps 0,1,4,5: U = U~ - W S_j as bf16 hi | lo, then thread 0 issues
//                  MMA 2 (M=128, N=64, K=64): [Da | Db] = Kr^T [U_hi | U_lo]
//   all:           S_{j+1} = Gamma_L(j) S_j + Da + Db in registers: the bf16
//                  operand, and a snapshot if chunk j ends at one
// The chunk-to-chunk chain is MMA 1 -> U -> MMA 2 -> state write-back; the
// output product, its store and the copies run beside it.  Records are
// prefetched two chunks ahead with bulk copies (TMA engine).  TMEM holds
// 3 x 64 columns of output accumulators and 64 of state.  The math is stated
// in kda_tc_common.cuh.
#pragma once

#include "kda_tc_handoff.cuh"

namespace kda {
namespace tcp {
namespace {

using namespace tc;

constexpr int kNh = 16;                 // state columns per thread
constexpr uint32_t kSopSbo = 16 * 128;  // S operand: 16 K-groups (key channels) per MN-group
constexpr uint32_t kUopSbo = 8 * 128;   // U operand: 8 K-groups (tokens) per MN-group
constexpr int kMmaThread = 0, kOutThread = 64, kLoadThread = 96;
constexpr int kUBarrier = 1;            // named barrier of the U warps
constexpr uint32_t kAqBytes = 64 * 64 * 2;

// A CTA carries NS = 32 or 64 state columns of one (sequence, head): 8 NS
// threads, two warps per TMEM lane quarter and column group of 16.  Every
// MMA runs at N = 2 NS (hi | lo); a tcgen05.mma costs about the same for
// any N <= 64 and little more at N = 128, so 64 columns per CTA take nearly
// the time of 32 per chain step on half the SMs.
// kSplit: one operand slot (the CTA then fits beside an intra-chunk CTA on
// one SM, as in the fused kernel), each chunk's operands copied in two
// parts as their areas free up: part A (AW, Gamma_L) once MMA 1 of the
// chunk before has read AW, part B (AK, U~) once its MMA 2 has read AK.
template <int NS, bool kSplit = false>
struct K3Cfg {
  static constexpr int kNop = 2 * NS;           // MMA N: hi and lo halves side by side
  static constexpr int kThreads = 8 * NS;       // 256 or 512
  static constexpr int kSlices = 128 / NS;      // column slices of a 128-column state
  static constexpr int kUThreads = 4 * NS;      // threads of the U warps (TMEM lanes 0-63)
  static constexpr uint32_t kTmemCols = 4 * kNop;
  // ring of chain operands: AW (32 KB) | AK (16 KB) | UT slice | GL
  static constexpr uint32_t AW = 0;
  static constexpr uint32_t AK = AW + 128 * 128 * 2;
  static constexpr uint32_t UT = AK + 128 * 64 * 2;
  static constexpr uint32_t GL = UT + 64 * NS * 4;
  static constexpr uint32_t SLOT = GL + 128 * 4;
  static constexpr int kSlots = kSplit ? 1 : NS == 32 ? 3 : 2;
  static constexpr int kFullBars = kSplit ? 2 : kSlots;  // (kSplit) parts A and B
  static constexpr uint32_t SOP = kSlots * SLOT;  // S operand [hi | lo], MN-major (n, c)
  // ring of A_qk tiles; each is read as rows 64-127 of an M=128 tile that
  // starts 1 KB before it, inside the S operand or the tile before
  static constexpr int kAqSlots = kSplit ? 2 : 3;
  static constexpr uint32_t AQ0 = SOP + kNop * 128 * 2;
  // two U operands [hi | lo], MN-major (n, i)
  static constexpr uint32_t U_BYTES = kNop * 64 * 2;
  static constexpr uint32_t U0 = AQ0 + kAqSlots * kAqBytes;
  static constexpr uint32_t BYTES = U0 + 2 * U_BYTES;
  static constexpr uint32_t TILES = UT;  // AW | AK, contiguous in the record too
  static constexpr uint32_t TX = TILES + 64 * NS * 4 + 128 * 4;
  static constexpr uint32_t TX_A = AK - AW + 128 * 4;       // AW, Gamma_L
  static constexpr uint32_t TX_B = UT - AK + 64 * NS * 4;   // AK, U~ slice
  static_assert(AK - AW == Rec::AK - Rec::AW, "AW | AK keep the record's layout");
  static_assert(SLOT % 16 == 0 && AQ0 % 16 == 0 && U0 % 16 == 0,
                "bulk-copy destinations and operand tiles are 16-byte aligned");
  static_assert(AQ0 >= 1024, "the A_qk tile descriptor starts 1 KB early inside shared memory");
  // (two CTAs per SM: 228 KB less 1 KB of static and 1 KB of reserved
  // shared memory each)
  static_assert(BYTES <= (kSplit ? 114688u : 226u * 1024u),
                "fits one CTA per SM, or (kSplit) two per SM beside an intra-chunk CTA");
  static_assert(kThreads / 32 == 4 * (NS / kNh), "two warps per lane quarter and 16-column group");
};

// The chain operands of chunk cidx: three bulk copies (AW | AK, this CTA's
// slice of U~, Gamma_L) on one barrier.
template <int NS>
__device__ __forceinline__ void k3_load_chain(const ChunkParams& p, uint8_t* slot, uint64_t* bar,
                                              int64_t cidx, int h, int n0) {
  using C = K3Cfg<NS, false>;
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, C::TX);
  bulk_g2s(slot + C::AW, rec + Rec::AW, C::TILES, bar);
  bulk_g2s(slot + C::UT, rec + Rec::UT + (n0 / 4) * 64 * 16, 64 * NS * 4, bar);
  bulk_g2s(slot + C::GL, rec + Rec::GL, 128 * 4, bar);
}

// (kSplit) part A of chunk cidx's chain operands (AW, Gamma_L) and part B
// (AK, this CTA's slice of U~), each on its own barrier
template <int NS>
__device__ __forceinline__ void k3_load_part_a(const ChunkParams& p, uint8_t* slot, uint64_t* bar,
                                               int64_t cidx, int h) {
  using C = K3Cfg<NS, true>;
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, C::TX_A);
  bulk_g2s(slot + C::AW, rec + Rec::AW, C::AK - C::AW, bar);
  bulk_g2s(slot + C::GL, rec + Rec::GL, 128 * 4, bar);
}
template <int NS>
__device__ __forceinline__ void k3_load_part_b(const ChunkParams& p, uint8_t* slot, uint64_t* bar,
                                               int64_t cidx, int h, int n0) {
  using C = K3Cfg<NS, true>;
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, C::TX_B);
  bulk_g2s(slot + C::AK, rec + Rec::AK, C::UT - C::AK, bar);
  bulk_g2s(slot + C::UT, rec + Rec::UT + (n0 / 4) * 64 * 16, 64 * NS * 4, bar);
}

// The A_qk tile of chunk cidx.
__device__ __forceinline__ void k3_load_aq(const ChunkParams& p, uint8_t* dst, uint64_t* bar,
                                           int64_t cidx, int h) {
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, kAqBytes);
  bulk_g2s(dst, rec + Rec::AQ, kAqBytes, bar);
}

// This thread's 16 columns of a hi | lo accumulator pair, summed: v[n] =
// column (h16 + n) + column (NS + h16 + n) of one TMEM lane.
template <int NS>
__device__ __forceinline__ void tmem_ld_sum(uint32_t taddr, int h16, float* v) {
  float b[kNh];
  tmem_ld16(taddr + h16, v);
  tmem_ld16(taddr + NS + h16, b);
  tmem_ld_wait();
#pragma unroll
  for (int n = 0; n < kNh; ++n) v[n] += b[n];
}

// bf16 hi and lo parts of 8 fp32 values, packed
__device__ __forceinline__ void split8(const float* u, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    h[t] = pack_bf16(u[2 * t], u[2 * t + 1]);
    l[t] = pack_bf16(u[2 * t] - bf16_lo(h[t]), u[2 * t + 1] - bf16_hi(h[t]));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// The output gate's logits of one o row (token i of chunk ch, head h, this
// thread's 16 columns; with a gate per head its one logit in r[0].x).  They
// are read two steps before the row is stored and turned into factors one
// step before, in the window where these warps wait for U and MMA 2, so the
// store itself only multiplies.
struct GateRow {
  uint4 r[kNh / 8];
};
struct GateF {
  float f[kNh];
};
__device__ __forceinline__ GateF gate_factors(const ChunkParams& p, const GateRow& g) {
  GateF x;
  if (p.out_gate_per_head) {
    const float f = gate_fast(bf16_lo(g.r[0].x));
#pragma unroll
    for (int n = 0; n < kNh; ++n) x.f[n] = f;
  } else {
#pragma unroll
    for (int q8 = 0; q8 < kNh / 8; ++q8)
#pragma unroll
      for (int j = 0; j < 8; ++j) x.f[8 * q8 + j] = gate_fast(bf16_at(g.r[q8], j));
  }
  return x;
}
__device__ __forceinline__ GateRow load_gate_row(const ChunkParams& p, const Chunk& ch, int i, int h,
                                                 int n0, int h16) {
  GateRow g{};
  if (p.out_gate && i < ch.len && p.k3_mode != kScanPass1) {
    const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(p.out_gate);
    const int64_t row = (ch.tok0 + i) * p.H + h;
    if (p.out_gate_per_head) {
      g.r[0].x = (uint32_t)__bfloat16_as_ushort(r[row]);
    } else {
      const uint4* rg = reinterpret_cast<const uint4*>(r + row * (int64_t)p.dv + n0 + h16);
#pragma unroll
      for (int q8 = 0; q8 < kNh / 8; ++q8) g.r[q8] = __ldg(rg + q8);
    }
  }
  return g;
}

// o rows of one chunk from lanes 64-127 of an output accumulator: row i, this
// thread's 16 columns (none in the first pass of the segment scan), times
// the output gate's factors gf when there is a gate.  The TMEM read is
// warp-collective: every lane takes it; only lanes whose waits succeeded
// (`live`) store.
template <int NS>
__device__ __forceinline__ void store_output(const ChunkParams& p, const Chunk& ch, uint32_t d1,
                                             int h16, int i, int h, int n0, const GateF& gf, bool live) {
  float d[kNh];
  tmem_ld_sum<NS>(d1, h16, d);
  if (live && i < ch.len && p.k3_mode != kScanPass1) {
    const float scale = p.scale;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
    const int64_t row = (ch.tok0 + i) * p.H + h;
    uint4* dst = reinterpret_cast<uint4*>(o + row * (int64_t)p.dv + n0 + h16);
    if (p.out_gate)
#pragma unroll
      for (int n = 0; n < kNh; ++n) d[n] *= gf.f[n];
#pragma unroll
    for (int q8 = 0; q8 < kNh / 8; ++q8)
      dst[q8] = make_uint4(pack_bf16(scale * d[8 * q8], scale * d[8 * q8 + 1]),
                           pack_bf16(scale * d[8 * q8 + 2], scale * d[8 * q8 + 3]),
                           pack_bf16(scale * d[8 * q8 + 4], scale * d[8 * q8 + 5]),
                           pack_bf16(scale * d[8 * q8 + 6], scale * d[8 * q8 + 7]));
  }
}

// The state operand of one key channel c, this thread's 16 columns: the
// bf16 [hi | lo] pair of v.
template <int NS>
__device__ __forceinline__ void write_operand(uint8_t* sop, int c, int h16, const float* v) {
#pragma unroll
  for (int m = 0; m < kNh / 8; ++m) {
    uint4 hi, lo;
    split8(v + 8 * m, hi, lo);
    *reinterpret_cast<uint4*>(sop + mnmajor_off(h16 + 8 * m, c, kSopSbo)) = hi;
    *reinterpret_cast<uint4*>(sop + mnmajor_off(NS + h16 + 8 * m, c, kSopSbo)) = lo;
  }
}

// The mbarriers of a chain CTA and its TMEM address
template <int NS, bool kSplit = false>
struct K3Bars {
  uint64_t full[K3Cfg<NS, kSplit>::kFullBars];
  uint64_t aq[K3Cfg<NS, kSplit>::kAqSlots];
  uint64_t mma1;     // MMA 1
  uint64_t mma2;     // MMA 2 (state chain)
  uint64_t mma3[2];  // MMA 3 of even / odd chunks (output path)
  uint64_t drain;    // every MMA, on the error path
  uint32_t tmem_base;
  // (kFused) the records of the chain's first `pub` chunks are published,
  // as thread kLoadThread found them; read by thread kOutThread after a
  // CTA barrier
  int64_t pub;
};

// The chain of (sequence s, head h, column slice z % kSlices) on a whole CTA
// of K3Cfg<NS>::kThreads threads with K3Cfg<NS>::BYTES of shared memory at sm.
// kPoll: the instantiation for wait limits under kPollLimitNs (the give-up
// test); NS: the state columns of a CTA (K3Cfg).  kFused: the records are
// made by the item pipelines of the fused kernel while the chain runs: a
// record is copied once it is published (kda_tc_handoff.cuh).  kSplit: one
// operand slot, copied in two parts (K3Cfg).
template <bool kPoll, int NS, bool kFused, bool kSplit = false>
__device__ __forceinline__ void inter_chain(const ChunkParams& p, int s, int h, int z, uint8_t* sm,
                                            K3Bars<NS, kSplit>& bars) {
  using C = K3Cfg<NS, kSplit>;
  constexpr int kNs = NS, kNop = C::kNop;
  uint64_t* const bar_full = bars.full;
  uint64_t* const bar_aq = bars.aq;
  uint64_t& bar_mma1 = bars.mma1;
  uint64_t& bar_mma2 = bars.mma2;
  uint64_t* const bar_mma3 = bars.mma3;
  uint64_t& bar_drain = bars.drain;
  uint32_t& tmem_base = bars.tmem_base;

  const int n0 = (z % C::kSlices) * kNs;
  // first pass of the segment scan: CTAs z >= kSlices carry the transition
  // map (identity state, U~ = 0), the others the state offset (zero state)
  const bool pass1 = p.k3_mode == kScanPass1;
  const bool trans = pass1 && z >= C::kSlices;
  const int H = p.H, tid = threadIdx.x, warp = tid >> 5;
  // (kFused, one operand ring: the overlapped schedule) this CTA started as
  // the programmatic dependent of the intra-chunk kernel, without waiting for
  // it; what it reads of the planning kernel's outputs was complete before
  // any intra-chunk CTA signalled (each waited for the planning kernel
  // first).  The scalars are read through L2.
  constexpr bool kOvl = kFused && !kSplit;
  const int64_t c_begin = kOvl ? __ldcg(p.seq_chunk_begin + s) : p.seq_chunk_begin[s];
  const int64_t c_end = kOvl ? __ldcg(p.seq_chunk_begin + s + 1) : p.seq_chunk_begin[s + 1];
  const int64_t total_chunks = kOvl ? __ldcg(&p.meta->total_chunks) : p.meta->total_chunks;
  if (c_end > c_begin && total_chunks == 0) return;  // chunk table overflowed
  const int64_t nchunks = c_end - c_begin;

  // TMEM lane quarter of this warp, its 16 columns, its key channel / token row
  const int quarter = warp & 3;
  const int h16 = (warp >> 2) * kNh;
  const int c = tid & 127;
  const bool u_warp = quarter < 2;  // warps 0, 1, 4, 5: lanes 0-63 (W rows, U)
  uint8_t* SOP = sm + C::SOP;

  if (warp == 0) tmem_alloc(&tmem_base, C::kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < C::kFullBars; ++i) mbar_init(&bar_full[i], 1);
    for (int i = 0; i < C::kAqSlots; ++i) mbar_init(&bar_aq[i], 1);
    mbar_init(&bar_mma1, 1);
    mbar_init(&bar_mma2, 1);
    mbar_init(&bar_mma3[0], 1);
    mbar_init(&bar_mma3[1], 1);
    mbar_init(&bar_drain, 2);  // the two MMA-issuing threads
    mbar_init_fence();
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)(32 * quarter) << 16;
  const uint32_t DS = tmem + 3 * kNop + lane_off;  // [Da | Db], lane = key channel
  // output accumulator of chunk j (this warp's lanes): [W;Qp] S_j, then
  // + A_qk U in lanes 64-127
  auto d1_of = [&](int64_t j) { return tmem + (uint32_t)(j % 3) * kNop; };
  auto slot_of = [&](int64_t j) { return sm + (uint32_t)(j % C::kSlots) * C::SLOT; };
  auto aq_of = [&](int64_t j) {
    return sm + C::AQ0 + (uint32_t)(j % C::kAqSlots) * kAqBytes;
  };
  auto u_of = [&](int64_t j) { return sm + C::U0 + (uint32_t)(j & 1) * C::U_BYTES; };
  // (the drain of the error path waits with the long limit; in the fused
  // kernel a copy may have been issued only once its record came, and its
  // wait takes the handoff's limit)
  const uint64_t copy_limit = kFused ? handoff_limit_ns(p) : p.wait_ns;
  // the chain operands of chunk j (kSplit: part A) have landed
  auto wait_chain = [&](int64_t j, bool drain) {
    uint64_t* bar = &bar_full[j % C::kSlots];
    const uint32_t par = (uint32_t)((j / C::kSlots) & 1);
    return drain ? mbar_wait(bar, par, kWaitLimitNs) : mbar_wait_t<kPoll>(bar, par, copy_limit);
  };
  // (kSplit) part B of chunk j has landed
  auto wait_part_b = [&](int64_t j, bool drain) {
    uint64_t* bar = &bar_full[kSplit ? 1 : 0];
    const uint32_t par = (uint32_t)(j & 1);
    return drain ? mbar_wait(bar, par, kWaitLimitNs) : mbar_wait_t<kPoll>(bar, par, copy_limit);
  };

  // Thread 96 issues the chain-operand copies (kSplit: both parts) and
  // thread 64 the A_qk copies, in chunk order; each counts what it issued
  // and what was waited for, so the error path can let copies in flight
  // land.  (kFused) A copy is issued once its record is published: where its
  // area frees up before that, the copy is left for later (`now` false) and
  // issued, waiting for the record, just before the chunk is needed.  False
  // only if that wait gave up.
  int64_t chain_issued = 0, chain_waited = 0, aq_issued = 0, aq_waited = 0;
  int64_t b_issued = 0, b_waited = 0;  // (kSplit) part B
  bool ok = true;
  bool okl = true;  // this thread's own waits succeeded
  // (kFused) record j is published, as seen by this thread (an acquire,
  // then a proxy fence before the copies that read it): 1 yes, 0 not yet
  // (`now` false: no wait), -1 the wait gave up.  The records of chunks
  // below `pub` are known published.  Thread kLoadThread, finding record j
  // not known, reads the flags of up to kScanAhead chunks from `pub` on at
  // once (relaxed loads in flight together) and takes the published ones in
  // order with one acquire fence: an acquire load per record would hold its
  // warp, which also takes part in every chain step, for a round trip to L2
  // each time.  It leaves `pub` in shared memory, where thread kOutThread
  // takes it after the next CTA barrier.
  constexpr int kScanAhead = 16;
  int64_t pub = 0;
  if (kFused && tid == kLoadThread) bars.pub = 0;
  auto ready = [&](int64_t j, bool now) -> int {
    if constexpr (kFused) {
      if (j < pub) return 1;
      if (tid == kLoadThread && !now) {
        // batches of kScanAhead flags, while a whole batch is published
        int64_t q = pub;
        for (;;) {
          uint32_t f[kScanAhead];
#pragma unroll
          for (int k = 0; k < kScanAhead; ++k)
            f[k] = q + k < nchunks ? ld_relaxed_u32(rec_flag(p, c_begin + q + k, h)) : 0u;
          int n = 0;
          while (n < kScanAhead && f[n] != 0u) ++n;
          q += n;
          if (n < kScanAhead) break;
        }
        if (q > pub) {
          fence_gpu();  // with the relaxed loads that saw the flags: an acquire
          fence_proxy_async_global();
          pub = q;
          *reinterpret_cast<volatile int64_t*>(&bars.pub) = pub;
        }
        return j < pub ? 1 : 0;
      }
      if (!now) return 0;
      if (!rec_wait_published(p, c_begin + j, h)) return -1;
      if (j == pub) {
        pub = j + 1;
        if (tid == kLoadThread) *reinterpret_cast<volatile int64_t*>(&bars.pub) = pub;
      }
    }
    return 1;
  };
  auto issue_chain = [&](int64_t j, bool now) -> bool {
    const int r = ready(j, now);
    if (r <= 0) return r == 0;
    if constexpr (kSplit)
      k3_load_part_a<NS>(p, slot_of(j), &bar_full[0], c_begin + j, h);
    else
      k3_load_chain<NS>(p, slot_of(j), &bar_full[j % C::kSlots], c_begin + j, h, n0);
    chain_issued = j + 1;
    return true;
  };
  auto issue_b = [&](int64_t j, bool now) -> bool {
    if constexpr (kSplit) {
      const int r = ready(j, now);
      if (r <= 0) return r == 0;
      k3_load_part_b<NS>(p, slot_of(j), &bar_full[1], c_begin + j, h, n0);
      b_issued = j + 1;
    }
    return true;
  };
  auto issue_aq = [&](int64_t j, bool now) -> bool {
    const int r = ready(j, now);
    if (r <= 0) return r == 0;
    k3_load_aq(p, aq_of(j), &bar_aq[j % C::kAqSlots], c_begin + j, h);
    aq_issued = j + 1;
    return true;
  };
  if (tid == kLoadThread) {
    // (kFused) the first scan of the flags before any copy is issued: its
    // acquire fence then waits behind none
    if (kFused && nchunks > 0) ready(0, false);
    for (int64_t j = 0; okl && j < C::kSlots && j < nchunks && chain_issued == j; ++j)
      okl = issue_chain(j, j == 0);
    if (kSplit && okl && nchunks > 0) okl = issue_b(0, true);
  }
  if (tid == kOutThread)
    for (int64_t j = 0; okl && j < C::kAqSlots && j < nchunks && aq_issued == j; ++j)
      okl = issue_aq(j, kFused && j == 0);
  // initial state: the operand holds S_0, TMEM Gamma_L(0) S_0.  States are
  // [dk][dv] in global memory; a head narrower than 128 channels (dk or dv =
  // 64) runs zero-padded: key rows c >= dk hold zeros and are never written,
  // and the grid covers only the dv / kNs column slices that exist.
  const int DK = p.dk, DV = p.dv;
  const bool row_live = c < DK;
  const size_t sbase = ((size_t)s * H + h) * DK * DV;
  float sreg[kNh];  // this thread's 16 state values (key channel c), fp32
  {
    float v[kNh];
#pragma unroll
    for (int n = 0; n < kNh; n += 4) {
      float4 x = p.initial_state && !pass1 && row_live
                     ? *reinterpret_cast<const float4*>(p.initial_state + sbase + (size_t)c * DV + n0 + h16 + n)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      v[n] = x.x; v[n + 1] = x.y; v[n + 2] = x.z; v[n + 3] = x.w;
    }
    if (trans)
#pragma unroll
      for (int n = 0; n < kNh; ++n) v[n] = c == n0 + h16 + n ? 1.f : 0.f;
#pragma unroll
    for (int n = 0; n < kNh; ++n) sreg[n] = v[n];
    write_operand<NS>(SOP, c, h16, v);
  }

  const uint32_t id = idesc_bf16(128, kNop, 0, 1);     // B operands MN-major
  const uint32_t id_ak = idesc_bf16(128, kNop, 1, 1);  // Kr^T is MN-major too
  // MMA 3 of chunk j, thread 64: wait for its A_qk tile, then
  // D1[j % 3] += A_qk [U_hi | U_lo].  False if the tile never came.
  auto mma3 = [&](int64_t j) -> bool {
    // (kFused) a tile left for later is copied now: its slot's last tile,
    // chunk j - kAqSlots's, was read by an MMA 3 awaited a step ago
    if (aq_issued == j && !issue_aq(j, true)) return false;
    if (!mbar_wait_t<kPoll>(&bar_aq[j % C::kAqSlots], (uint32_t)((j / C::kAqSlots) & 1), copy_limit))
      return false;
    aq_waited = j + 1;
    const uint32_t a = smem_u32(aq_of(j)) - 1024, ub = smem_u32(u_of(j));
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mma_bf16(d1_of(j), sdesc(a + k * 2 * 1024, 1024, 128), sdesc(ub + k * 256, 128, kUopSbo), id, 1);
    mma_commit(&bar_mma3[j & 1]);
    return true;
  };
  // MMA 3 of chunk j completes phase j / 2 of bar_mma3[j & 1].  Its waiters
  // are done before the next commit to that barrier (two steps later, behind
  // a CTA barrier), so a parity wait never sees two phases complete.
  auto wait_mma3 = [&](int64_t j) {
    return mbar_wait_t<kPoll>(&bar_mma3[j & 1], (uint32_t)((j >> 1) & 1), p.wait_ns);
  };

  uint32_t ph1 = 0, ph2 = 0;
  Chunk prev1{}, prev2{};
  GateRow graw{};   // the output gate's logits of chunk it-1's row (read last step)
  GateF gfac{};     // its factors for chunk it-2's row (formed last step)
  Chunk next = nchunks > 0 ? p.chunks[c_begin] : Chunk{};
  for (int64_t it = 0; it < nchunks; ++it) {
    uint8_t* slot = slot_of(it);
    uint8_t* uop = u_of(it);
    const Chunk ch = next;  // chunk entries are read one step ahead
    if (it + 1 < nchunks) next = p.chunks[c_begin + it + 1];
    // this chunk's operands (kFused: copied now if their record came late;
    // kSplit: part B too) have landed; Gamma_L(it) is read before any copy
    // can take the slot (kSplit: part A of chunk it+1, during this step)
    if (kFused && tid == kLoadThread && okl && chain_issued == it) okl = issue_chain(it, true);
    if (kSplit && tid == kLoadThread && okl && b_issued == it) okl = issue_b(it, true);
    okl = okl && wait_chain(it, false);
    if (okl) chain_waited = it + 1;  // a copy still in flight is left to the drain
    const float gl_cur = reinterpret_cast<const float*>(slot_of(it) + C::GL)[c];
    // the state operand of this step is written
    fence_async_smem();
    fence_before_sync();
    ok = __syncthreads_and(okl);
    fence_after_sync();
    if (!ok) break;
    if (kFused && tid == kOutThread) {
      const int64_t q = *reinterpret_cast<volatile int64_t*>(&bars.pub);
      if (q > pub) {
        pub = q;
        fence_proxy_async_global();  // before its copies read those records
      }
    }
    // (kFused, kSplit) a first look at chunk it+1's record, early: its part
    // A can then go in as soon as MMA 1 has read AW
    if (kFused && kSplit && tid == kLoadThread && okl && it + 1 < nchunks) ready(it + 1, false);
    if (tid == kMmaThread) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(d1_of(it), sdesc(smem_u32(slot + C::AW) + k * 2 * 128 * 16, 128 * 16, 128),
                 sdesc(smem_u32(SOP) + k * 256, 128, kSopSbo), id, k > 0);
      mma_commit(&bar_mma1);
    }
    if (!u_warp) {
      // the outputs of chunk it-2, whose MMA 3 was issued last step ...
      if (it >= 2) {
        okl = okl && wait_mma3(it - 2);
        fence_after_sync();
        store_output<NS>(p, prev2, d1_of(it - 2) + lane_off, h16, c - 64, h, n0, gfac, okl);
        // ... its A_qk tile takes chunk it+1 (with two tiles, chunk it, whose
        // slot held chunk it-2's) ...
        constexpr int kAqLead = C::kAqSlots - 2;
        if constexpr (kFused && !kSplit) {
          // (records that come late) every tile not yet copied whose slot is
          // free, in order, as far as their records are published
          if (tid == kOutThread)
            while (okl && aq_issued <= it + kAqLead && aq_issued < nchunks) {
              const int64_t j = aq_issued;
              okl = issue_aq(j, false);
              if (aq_issued == j) break;
            }
        } else {
          if (tid == kOutThread && okl && it + kAqLead < nchunks && aq_issued == it + kAqLead)
            okl = issue_aq(it + kAqLead, false);
        }
      }
      // ... with a 3-slot ring the slot of chunk it-1 (MMA 2 done) takes
      // chunk it+2 here, off the chain ...
      if constexpr (kFused && C::kSlots == 3) {
        // (records that come late) every chunk not yet copied whose slot is
        // free (up to chunk it+2), in order, as far as their records are
        // published; one still missing is copied, waiting, in the write-back
        // of the step before it is needed
        if (tid == kLoadThread && it >= 1)
          while (okl && chain_issued <= it + 2 && chain_issued < nchunks) {
            const int64_t j = chain_issued;
            okl = issue_chain(j, false);
            if (chain_issued == j) break;
          }
      } else {
        if (C::kSlots == 3 && tid == kLoadThread && okl && it >= 1 && it + 2 < nchunks) okl = issue_chain(it + 2, true);
      }
      // ... (kSplit) part A of chunk it+1 goes in once MMA 1 has read AW
      // (kFused: if its record was seen above) ...
      if (kSplit && tid == kLoadThread && okl && it + 1 < nchunks && chain_issued == it + 1 &&
          (!kFused || pub > it + 1)) {
        okl = mbar_wait_t<kPoll>(&bar_mma1, ph1, p.wait_ns);
        if (okl) okl = issue_chain(it + 1, false);
      }
      // ... and the output product of chunk it-1 runs once MMA 1 is done; the
      // gate logits of its row are fetched now, for its store next step
      if (tid == kOutThread && it >= 1 && okl) {
        okl = mbar_wait_t<kPoll>(&bar_mma1, ph1, p.wait_ns);
        if (okl) okl = mma3(it - 1);
      }
      if (p.out_gate) {  // factors of chunk it-1's row; logits of chunk it's row
        gfac = gate_factors(p, graw);
        graw = load_gate_row(p, ch, c - 64, h, n0, h16);
      }
    } else {
      // U = U~ - W S_j for token i = lane row, this thread's 16 columns.  The
      // U buffer of this step was last read by MMA 3 of chunk it-2, issued by
      // another thread: its completion is awaited too.
      okl = okl && mbar_wait_t<kPoll>(&bar_mma1, ph1, p.wait_ns);
      if (it >= 2) okl = okl && wait_mma3(it - 2);
      if constexpr (kSplit) {  // this chunk's U~ (part B)
        okl = okl && wait_part_b(it, false);
        if (okl) b_waited = it + 1;
      }
      fence_after_sync();
      const int i = c;
      float d[kNh];
      tmem_ld_sum<NS>(d1_of(it) + lane_off, h16, d);
      const float* ut = reinterpret_cast<const float*>(slot + C::UT);
      const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int m = 0; m < kNh / 8; ++m) {
        const int e = h16 + 8 * m;  // first of 8 columns
        const float4 ua = trans ? zero4 : *reinterpret_cast<const float4*>(ut + ((e / 4) * 64 + i) * 4);
        const float4 ub = trans ? zero4 : *reinterpret_cast<const float4*>(ut + ((e / 4 + 1) * 64 + i) * 4);
        const float u[8] = {ua.x - d[8 * m], ua.y - d[8 * m + 1], ua.z - d[8 * m + 2],
                            ua.w - d[8 * m + 3], ub.x - d[8 * m + 4], ub.y - d[8 * m + 5],
                            ub.z - d[8 * m + 6], ub.w - d[8 * m + 7]};
        uint4 hi, lo;
        split8(u, hi, lo);
        *reinterpret_cast<uint4*>(uop + mnmajor_off(e, i, kUopSbo)) = hi;
        *reinterpret_cast<uint4*>(uop + mnmajor_off(kNs + e, i, kUopSbo)) = lo;
      }
      fence_async_smem();
      asm volatile("bar.sync %0, %1;" ::"n"(kUBarrier), "n"(C::kUThreads) : "memory");
      // MMA 2, the state chain: [Da | Db] = Kr^T [U_hi | U_lo]
      if (tid == kMmaThread) {
        const uint32_t ub = smem_u32(uop);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(DS - lane_off, sdesc(smem_u32(slot + C::AK) + k * 256, 128, Rec::kAkSbo),
                   sdesc(ub + k * 256, 128, kUopSbo), id_ak, k > 0);
        mma_commit(&bar_mma2);
      }
    }
    ph1 ^= 1;
    // the state write-back: S_{j+1} = Gamma_L(j) S_j + Da + Db
    okl = okl && mbar_wait_t<kPoll>(&bar_mma2, ph2, p.wait_ns);
    ph2 ^= 1;
    fence_after_sync();
    // with a 2-slot ring, this chunk's slot takes chunk it+2 as soon as MMA 2
    // has read it (MMA 1 and the U warps before it; Gamma_L was read at the
    // step's top): a step of lead.  (kFused) only if its record is already
    // published; else it is copied before the wait for it at the top of its
    // step.
    if (C::kSlots == 2 && tid == kLoadThread && okl && it + 2 < nchunks && chain_issued == it + 2)
      okl = issue_chain(it + 2, false);
    // (kSplit) part B of chunk it+1 goes in now that MMA 2 has read AK and
    // the U warps have read U~ (before MMA 2 was issued), after part A
    // (thread 96 first waits for part B of chunk it itself, to keep its
    // barrier phases in step)
    if (kSplit && tid == kLoadThread && okl) {
      okl = wait_part_b(it, false);
      if (okl) {
        b_waited = it + 1;
        if (okl && it + 1 < nchunks && chain_issued == it + 2 && b_issued == it + 1) okl = issue_b(it + 1, false);
      }
    }
    {
      float v[kNh];
      tmem_ld_sum<NS>(DS, h16, v);
#pragma unroll
      for (int n = 0; n < kNh; ++n) {
        v[n] = fmaf(gl_cur, sreg[n], v[n]);
        sreg[n] = v[n];
      }
      if (ch.snap_slot >= 0 && p.snapshots && !pass1 && row_live) {
        float* dst = p.snapshots + ((size_t)ch.snap_slot * H + h) * DK * DV + (size_t)c * DV + n0 + h16;
#pragma unroll
        for (int n = 0; n < kNh; n += 4)
          *reinterpret_cast<float4*>(dst + n) = make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
      }
      write_operand<NS>(SOP, c, h16, v);
    }
    prev2 = prev1;
    prev1 = ch;
  }
  // the output products still open: chunk n-2 (issued) and chunk n-1 (not yet)
  fence_before_sync();
  ok = __syncthreads_and(ok && okl);
  fence_after_sync();
  if (ok && nchunks >= 1) {
    if (tid == kOutThread) okl = mma3(nchunks - 1);
    if (!u_warp) {
      if (nchunks >= 2) {
        okl = okl && wait_mma3(nchunks - 2);
        fence_after_sync();
        store_output<NS>(p, prev2, d1_of(nchunks - 2) + lane_off, h16, c - 64, h, n0, gfac, okl);
      }
      if (p.out_gate) gfac = gate_factors(p, graw);  // chunk n-1's row
      okl = okl && wait_mma3(nchunks - 1);
      fence_after_sync();
      store_output<NS>(p, prev1, d1_of(nchunks - 1) + lane_off, h16, c - 64, h, n0, gfac, okl);
    }
  }
  fence_before_sync();
  ok = __syncthreads_and(ok && okl);
  fence_after_sync();
  float* const fin = trans ? p.trans : p.final_state;
  if (ok && fin && row_live) {
    float* dst = fin + sbase + (size_t)c * DV + n0 + h16;
#pragma unroll
    for (int n = 0; n < kNh; n += 4)
      *reinterpret_cast<float4*>(dst + n) = make_float4(sreg[n], sreg[n + 1], sreg[n + 2], sreg[n + 3]);
  }
  if (!ok) {
    // let the copies and MMAs still in flight finish (each wait bounded)
    // before the shared memory and TMEM are given back
    if (tid == 0) flag(p.status, kFlagTimeout);
    if (tid == kLoadThread) {
      for (int64_t j = chain_waited; j < chain_issued; ++j) wait_chain(j, true);
      for (int64_t j = b_waited; j < b_issued; ++j) wait_part_b(j, true);
    }
    if (tid == kOutThread)
      for (int64_t j = aq_waited; j < aq_issued; ++j)
        mbar_wait(&bar_aq[j % C::kAqSlots], (uint32_t)((j / C::kAqSlots) & 1), kWaitLimitNs);
    if (tid == kMmaThread || tid == kOutThread) mma_commit(&bar_drain);
    if (tid == kMmaThread) mbar_wait(&bar_drain, 0, kWaitLimitNs);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
}

}  // namespace
}  // namespace tcp
}  // namespace kda
