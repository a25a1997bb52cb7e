// kda_tc_fused.cu -- the fused tensor-core prefill: the intra-chunk step and
// the inter-chunk chains of one call in one kernel, each chain reading the
// records of its (sequence, head) as the item pipelines publish them
// (kda_tc_handoff.cuh), from L2, a few chunks behind ("Kimi K3: The Manos,
// The Mythos, The Legendos", bullet list: FlashKDA's unrolling in chunks
// with a linear prefill; the chunked form is stated in kda_tc_common.cuh).
//
// Two CTAs of 256 threads per SM.  CTAs 0 .. grid-n_chain-1 each run one
// item pipeline (kda_tc_intra.cuh), the pipelines together taking the
// (chunk, head) items in order: item i = cidx * H + h goes to pipeline
// i mod (item CTAs), so the chunk levels come out in order, as the chains
// read them.  The last n_chain CTAs each run the chain of one (sequence,
// head, 32-column slice of the state) (kda_tc_inter.cuh, K3Cfg<32, true>:
// one operand slot, copied in two parts).  A chain CTA and an item CTA each
// take half an SM (about 111 KB of shared memory, 256 TMEM columns, 128
// registers a thread), so a chain shares its SM with a pipeline, whose
// CUDA-core work fills the issue slots that the chain's MMA waits leave idle.
// (A chain of 64 columns needs 217 KB, a whole SM; and two pipelines in one
// 512-thread CTA address their halves of the shared memory through a base
// held in registers, which costs them registers they do not have.)
#include "kda_tc_inter.cuh"
#include "kda_tc_intra.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int kChainNs = 32;  // state columns of a chain CTA
using ChainCfg = K3Cfg<kChainNs, true>;
constexpr uint32_t kFusedBytes = Smem::BYTES > ChainCfg::BYTES ? Smem::BYTES : ChainCfg::BYTES;
static_assert(ChainCfg::kThreads == kThreads, "a chain CTA and an item CTA have the same thread count");

template <bool kHeadGate, bool kConv>
__global__ void __launch_bounds__(kThreads, 2)
tc_fused(ChunkParams p, int64_t n_items, int32_t n_chain, const __grid_constant__ RowMaps maps) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ K3Bars<kChainNs, true> cbars;
  __shared__ IntraBars ibars;
  __shared__ uint32_t tmem_base;
  // two waves of `wave` CTAs; the last chain_sms slots of each wave are
  // chains, so that (CTAs being placed one per SM in index order, then a
  // second per SM) the chains pair up on chain_sms SMs and the pipelines on
  // the rest
  const int wave = (int)gridDim.x / 2, chain_sms = (n_chain + 1) / 2;
  const int b = (int)blockIdx.x, w = b / wave, slot = b % wave, pipe_slots = wave - chain_sms;
  if (slot >= pipe_slots) {
    const int ch = w * chain_sms + (slot - pipe_slots);
    if (ch >= n_chain) return;
    const int slices = p.dv / kChainNs, per_seq = p.H * slices;
    inter_chain<false, kChainNs, true, true>(p, ch / per_seq, (ch % per_seq) / slices, ch % slices, sm, cbars);
    return;
  }
  const int pipe = w * pipe_slots + slot;
  const int tid = threadIdx.x;
  if (tid < 32) tmem_alloc(&tmem_base, 256);
  if (tid == 0) init_intra_bars(&ibars);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (pipe < n_items)
    intra_items<false, kHeadGate, kConv, true>(
        p, maps, IntraPipe{sm, &ibars, tmem_base, tid, PipeSync{0}, (int64_t)pipe, 2 * (int64_t)pipe_slots, n_items});
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tmem_base, 256);
}

using FusedKernel = void (*)(ChunkParams, int64_t, int32_t, RowMaps);

cudaError_t set_fused_attributes(FusedKernel k) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedBytes);
}

FusedKernel fused_kernel(const ChunkParams& p) {
  const bool head = p.gate_per_head != 0, conv = p.conv_width > 0;
  return conv ? (head ? tc_fused<true, true> : tc_fused<false, true>)
              : (head ? tc_fused<true, false> : tc_fused<false, false>);
}

}  // namespace
}  // namespace tcp

int fused_chain_columns() { return tcp::kChainNs; }

// Two CTAs per SM: each takes kFusedBytes of dynamic shared memory, 1 KB of
// static (the alignment of the dynamic array) and 1 KB the system reserves
bool fused_supported(int device) {
  int smem = 0;
  if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess)
    return false;
  return (int64_t)smem >= 2 * ((int64_t)tcp::kFusedBytes + 2048);
}

cudaError_t launch_tc_fused(const ChunkParams& p, int32_t n_chain, int32_t grid, cudaStream_t stream) {
  using namespace tcp;
  // the record flags are the caller's (kda_api.cu): never launch without them
  if (!p.rec_ready || !p.inter || n_chain <= 0 || grid % 2 != 0 || n_chain > grid / 2) return cudaErrorInvalidValue;
  const FusedKernel kernel = fused_kernel(p);
  cudaError_t e = set_fused_attributes(kernel);
  if (e != cudaSuccess) return e;
  RowMaps maps;
  if (!make_row_maps(p, &maps)) return cudaErrorInvalidValue;
  const int64_t n_items = p.max_chunks * (int64_t)p.H;
  kernel<<<(unsigned)grid, kThreads, kFusedBytes, stream>>>(p, n_items, n_chain, maps);
  return cudaGetLastError();
}

}  // namespace kda
