// kda_tc_inter.cu -- K3, the inter-chunk kernel of the tensor-core prefill,
// and the launcher of the whole tensor-core prefill (K2 then K3).
//
// One CTA per (sequence, head, 32-column slice of S), walking the sequence's
// chunks in order.  The state slice lives in TMEM as an fp32 accumulator
// (lane = key channel); a bf16 copy of it in shared memory is the MMA
// operand.  Per chunk:
//   MMA 1 (M=128, N=32, K=128): [W S0 ; Qp S0]                 -> TMEM D1[b]
//   meanwhile: S <- Diag(Gamma_L) S with tcgen05.ld / st, and the output
//              rows of the previous chunk are read from D1[1-b]
//   threads: U = U~ - W S0 as a bf16 hi + lo pair
//   MMA 2/3 (M=128, N=32, K=64): S += Kr^T U,  D1[b][64..127] += A_qk U
//   threads: new bf16 state operand; snapshot
// The state and U operands are stored MN-major, so each thread writes its
// row as 16-byte chunks.  Records are prefetched two chunks ahead with bulk
// copies (TMA engine).  The math is stated in kda_tc_common.cuh.
#include "kda_tc_common.cuh"

namespace kda {
namespace tcp {
namespace {

using namespace tc;

constexpr int kThreads = 128;
constexpr int kNs = 32;                 // state columns per CTA
constexpr uint32_t kSopSbo = 16 * 128;  // S operand: 16 K-groups (key channels) per MN-group
constexpr uint32_t kUopSbo = 8 * 128;   // U operand: 8 K-groups (tokens) per MN-group

struct K3Smem {
  // one ring slot: AW (32 KB) | AK (16 KB) | AQ128 (16 KB, rows 64-127 used) | UT slice | GL
  static constexpr uint32_t AW = 0;
  static constexpr uint32_t AK = AW + 128 * 128 * 2;
  static constexpr uint32_t AQ = AK + 128 * 64 * 2;
  static constexpr uint32_t UT = AQ + 128 * 64 * 2;
  static constexpr uint32_t GL = UT + 64 * kNs * 4;
  static constexpr uint32_t SLOT = GL + 128 * 4;
  static constexpr uint32_t SOP = 2 * SLOT;              // S operand, MN-major (n, c)
  static constexpr uint32_t UHI = SOP + kNs * 128 * 2;    // U operand, MN-major (n, i)
  static constexpr uint32_t ULO = UHI + kNs * 64 * 2;
  static constexpr uint32_t BYTES = ULO + kNs * 64 * 2;
  static constexpr uint32_t TILES = UT;  // AW | AK | AQ, contiguous in the record too
  static constexpr uint32_t TX = TILES + 64 * kNs * 4 + 128 * 4;
};
static_assert(K3Smem::AK - K3Smem::AW == Rec::AK - Rec::AW &&
                  K3Smem::AQ - K3Smem::AW == Rec::AQ - Rec::AW &&
                  K3Smem::UT - K3Smem::AW == Rec::UT - Rec::AW,
              "the operand tiles keep the record's relative layout");

// Three bulk copies per chunk: the operand tiles (64 KB), this CTA's slice of
// U~ and Gamma_L.
__device__ __forceinline__ void k3_issue_loads(const ChunkParams& p, uint8_t* slot, uint64_t* bar,
                                               int64_t cidx, int h, int n0) {
  const uint8_t* rec = reinterpret_cast<const uint8_t*>(p.inter) + ((size_t)cidx * p.H + h) * Rec::BYTES;
  mbar_arrive_expect_tx(bar, K3Smem::TX);
  bulk_g2s(slot + K3Smem::AW, rec + Rec::AW, K3Smem::TILES, bar);
  bulk_g2s(slot + K3Smem::UT, rec + Rec::UT + (n0 / 4) * 64 * 16, 64 * kNs * 4, bar);
  bulk_g2s(slot + K3Smem::GL, rec + Rec::GL, 128 * 4, bar);
}

// 32 consecutive fp32 values of one TMEM lane (two 16-column loads)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  tmem_ld16(taddr, v);
  tmem_ld16(taddr + 16, v + 16);
  tmem_ld_wait();
}

// the S operand row of key channel c: 4 chunks of 8 bf16 (MN-major)
__device__ __forceinline__ void store_state_operand(uint8_t* sop, int c, const float* v) {
#pragma unroll
  for (int m = 0; m < kNs / 8; ++m)
    *reinterpret_cast<uint4*>(sop + mnmajor_off(8 * m, c, kSopSbo)) =
        make_uint4(pack_bf16(v[8 * m], v[8 * m + 1]), pack_bf16(v[8 * m + 2], v[8 * m + 3]),
                   pack_bf16(v[8 * m + 4], v[8 * m + 5]), pack_bf16(v[8 * m + 6], v[8 * m + 7]));
}

// o rows of one chunk from lanes 64-127 of an output accumulator (warps 2, 3)
__device__ __forceinline__ void store_output(const ChunkParams& p, const Chunk& ch, uint32_t d1,
                                             uint32_t lane_off, int i, int h, int n0) {
  float d[kNs];
  tmem_ld32(d1 + lane_off, d);
  if (i < ch.len) {
    const float scale = p.scale;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o);
    uint4* dst = reinterpret_cast<uint4*>(o + ((ch.tok0 + i) * p.H + h) * (int64_t)kD + n0);
#pragma unroll
    for (int q8 = 0; q8 < kNs / 8; ++q8)
      dst[q8] = make_uint4(pack_bf16(scale * d[8 * q8], scale * d[8 * q8 + 1]),
                           pack_bf16(scale * d[8 * q8 + 2], scale * d[8 * q8 + 3]),
                           pack_bf16(scale * d[8 * q8 + 4], scale * d[8 * q8 + 5]),
                           pack_bf16(scale * d[8 * q8 + 6], scale * d[8 * q8 + 7]));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
tc_inter(ChunkParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar_full[2];
  __shared__ __align__(8) uint64_t bar_mma;   // MMA 1 (one issuing thread)
  __shared__ __align__(8) uint64_t bar_mma2;  // MMA 2 (state chain)
  __shared__ __align__(8) uint64_t bar_mma3;  // MMA 3 (output path)
  __shared__ uint32_t tmem_base;

  const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * kNs;
  const int H = p.H, tid = threadIdx.x, warp = tid >> 5;
  const int64_t c_begin = p.seq_chunk_begin[s], c_end = p.seq_chunk_begin[s + 1];
  if (c_end > c_begin && p.meta->total_chunks == 0) return;  // chunk table overflowed
  const int64_t nchunks = c_end - c_begin;

  uint8_t* SOP = sm + K3Smem::SOP;
  uint8_t* UHI = sm + K3Smem::UHI;
  uint8_t* ULO = sm + K3Smem::ULO;

  if (warp == 0) tmem_alloc(&tmem_base, 128);
  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_mma2, 1);
    mbar_init(&bar_mma3, 1);
    mbar_init_fence();
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t D1[2] = {tmem, tmem + kNs};  // [W;Qp] S0, then + A_qk U in lanes 64-127
  const uint32_t DS = tmem + 2 * kNs;         // the state slice, lane = key channel
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
    store_state_operand(SOP, c, v);
  }

  const uint32_t id = idesc_bf16(128, kNs, 0, 1);     // B operands MN-major
  const uint32_t id_ak = idesc_bf16(128, kNs, 1, 1);  // Kr^T is MN-major too
  uint32_t mma_phase = 0, mma2_phase = 0, mma3_phase = 0;
  bool ok = true, ok3 = true;
  Chunk prev{};
  Chunk next = nchunks > 0 ? p.chunks[c_begin] : Chunk{};
  for (int64_t it = 0; it < nchunks && ok; ++it) {
    const int slot_i = (int)(it & 1), b = (int)(it & 1);
    uint8_t* slot = sm + slot_i * K3Smem::SLOT;
    const Chunk ch = next;  // chunk entries are read one step ahead
    if (it + 1 < nchunks) next = p.chunks[c_begin + it + 1];
    // S operand (previous iteration) and this slot are ready
    fence_async_smem();
    fence_before_sync();
    ok = __syncthreads_and(ok3 && mbar_wait(&bar_full[slot_i], (uint32_t)((it >> 1) & 1), kWaitLimitNs));
    fence_after_sync();
    if (!ok) break;
    if (tid == 0) {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mma_bf16(D1[b], sdesc(smem_u32(slot + K3Smem::AW) + k * 2 * 128 * 16, 128 * 16, 128),
                 sdesc(smem_u32(SOP) + k * 256, 128, kSopSbo), id, k > 0);
      mma_commit(&bar_mma);
    }
    // while MMA 1 runs: retention of the carried state, S <- Diag(Gamma_L) S ...
    {
      const float gl = reinterpret_cast<const float*>(slot + K3Smem::GL)[c];
      float v[kNs];
      tmem_ld32(DS + lane_off, v);
#pragma unroll
      for (int n = 0; n < kNs; ++n) v[n] *= gl;
      tmem_st16(DS + lane_off, v);
      tmem_st16(DS + lane_off + 16, v + 16);
      tmem_st_wait();
    }
    // ... and the outputs of the previous chunk
    if (it > 0 && warp >= 2) store_output(p, prev, D1[b ^ 1], lane_off, tid - 64, h, n0);
    fence_before_sync();
    ok = __syncthreads_and(mbar_wait(&bar_mma, mma_phase, kWaitLimitNs));
    mma_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    if (warp < 2) {
      // U = U~ - W S0 for token i = lane row, split into bf16 hi + lo
      const int i = tid;
      float d[kNs];
      tmem_ld32(D1[b] + lane_off, d);
      const float* ut = reinterpret_cast<const float*>(slot + K3Smem::UT);
#pragma unroll
      for (int m = 0; m < kNs / 8; ++m) {
        const float4 ua = *reinterpret_cast<const float4*>(ut + ((2 * m) * 64 + i) * 4);
        const float4 ub = *reinterpret_cast<const float4*>(ut + ((2 * m + 1) * 64 + i) * 4);
        const float u[8] = {ua.x - d[8 * m], ua.y - d[8 * m + 1], ua.z - d[8 * m + 2],
                            ua.w - d[8 * m + 3], ub.x - d[8 * m + 4], ub.y - d[8 * m + 5],
                            ub.z - d[8 * m + 6], ub.w - d[8 * m + 7]};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          hi[t] = pack_bf16(u[2 * t], u[2 * t + 1]);
          lo[t] = pack_bf16(u[2 * t] - bf16_lo(hi[t]), u[2 * t + 1] - bf16_hi(hi[t]));
        }
        *reinterpret_cast<uint4*>(UHI + mnmajor_off(8 * m, i, kUopSbo)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(ULO + mnmajor_off(8 * m, i, kUopSbo)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    // MMA 2, the state chain: S += Kr^T U; then MMA 3, the output path:
    // D1[b][64..127] += A_qk U (U as hi + lo).  Separate commits, so the
    // state write-back below waits for MMA 2 only and overlaps MMA 3.
    if (tid == 0) {
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t ub = smem_u32(part ? ULO : UHI);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(DS, sdesc(smem_u32(slot + K3Smem::AK) + k * 256, 128, Rec::kAkSbo),
                   sdesc(ub + k * 256, 128, kUopSbo), id_ak, 1);
      }
      mma_commit(&bar_mma2);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const uint32_t ub = smem_u32(part ? ULO : UHI);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_bf16(D1[b], sdesc(smem_u32(slot + K3Smem::AQ) + k * 2 * 128 * 16, 128 * 16, 128),
                   sdesc(ub + k * 256, 128, kUopSbo), id, 1);
      }
      mma_commit(&bar_mma3);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma2, mma2_phase, kWaitLimitNs));
    mma2_phase ^= 1;
    fence_after_sync();
    if (!ok) break;
    // new state: bf16 operand copy, snapshot if this chunk ends at one
    {
      float v[kNs];
      tmem_ld32(DS + lane_off, v);
      store_state_operand(SOP, c, v);
      if (ch.snap_slot >= 0 && p.snapshots) {
        float* dst = p.snapshots + ((size_t)ch.snap_slot * H + h) * kD * kD + (size_t)c * kD + n0;
#pragma unroll
        for (int n = 0; n < kNs; n += 4)
          *reinterpret_cast<float4*>(dst + n) = make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
      }
    }
    // warps 2-3 read the outputs of this chunk next step: after their state
    // rows are written back they wait for MMA 3, after which the slot is free
    // and a thread of warp 2 refills it with chunk it + 2
    if (warp >= 2) {
      ok3 = ok3 && mbar_wait(&bar_mma3, mma3_phase, kWaitLimitNs);
      fence_after_sync();
      if (tid == 64 && ok3 && it + 2 < nchunks)
        k3_issue_loads(p, slot, &bar_full[slot_i], c_begin + it + 2, h, n0);
    }
    mma3_phase ^= 1;
    prev = ch;
  }
  ok = __syncthreads_and(ok && ok3);
  fence_after_sync();
  if (ok && nchunks > 0 && warp >= 2)
    store_output(p, prev, D1[(nchunks - 1) & 1], lane_off, tid - 64, h, n0);
  if (!ok && tid == 0) flag(p.status, kFlagTimeout);
  if (p.final_state && ok) {
    float v[kNs];
    tmem_ld32(DS + lane_off, v);
    float* dst = p.final_state + sbase + (size_t)c * kD + n0;
#pragma unroll
    for (int n = 0; n < kNs; n += 4)
      *reinterpret_cast<float4*>(dst + n) = make_float4(v[n], v[n + 1], v[n + 2], v[n + 3]);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace
}  // namespace tcp

const bool kHaveTensorCorePath = true;

size_t tc_record_bytes() { return tcp::Rec::BYTES; }

cudaError_t launch_tc_prefill(const ChunkParams& p, cudaStream_t stream, cudaEvent_t mid) {
  using namespace tcp;
  cudaError_t e = launch_intra(p, stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tc_inter, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)K3Smem::BYTES);
  if (e != cudaSuccess) return e;
  if (mid) {
    e = cudaEventRecord(mid, stream);
    if (e != cudaSuccess) return e;
  }
  dim3 grid2((unsigned)p.num_seqs, (unsigned)p.H, (unsigned)(kD / kNs));
  tc_inter<<<grid2, kThreads, K3Smem::BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
