// kda_tc_overlap.cu -- the overlapped tensor-core prefill: the intra-chunk
// kernel (K2) and the inter-chunk kernel (K3) of one call, the chains of K3
// starting while K2 makes its last records ("Kimi K3: The Manos, The Mythos,
// The Legendos", bullet list: FlashKDA's unrolling in chunks with a linear
// prefill; the chunked form is stated in kda_tc_common.cuh).
//
// A chain of K3 runs serially over the chunks of its (sequence, head) and
// takes an SM of its own; K2 is throughput work over every (chunk, head)
// item.  Run one after the other, the chains start only once the last item
// is made, although a chain needs chunk j only j chain steps after it
// starts.  Here K2 runs on every SM, taking items in chunk order from a
// shared counter, until `ovl_split` items have been taken; then its CTAs
// leave, except those on `ovl_stay_sms` SMs (elected by the first K2 CTA to
// start on each SM), which take the remaining items.  K3 is launched as the
// programmatic dependent of K2 (every K2 CTA signals at its start), so its
// chain CTAs, each needing a whole SM, start on the SMs the leaving K2 CTAs
// free, and read each record once K2 has published it (kda_tc_handoff.cuh):
// from L2, a few chunks behind.  The split is set so that the staying SMs
// make the remaining records about as fast as the chains read them.
//
// Every wait ends: K3 starts only when every K2 CTA has started, K2 never
// waits for K3, and the staying K2 CTAs take every item left.  Records,
// flags and results are those of the separate kernels, bit for bit.
#include "kda_tc_inter.cuh"
#include "kda_tc_intra.cuh"

namespace kda {
namespace tcp {
namespace {

constexpr int kOvlNs = 32;  // state columns of a chain CTA
using OvlChainCfg = K3Cfg<kOvlNs, false>;

// (thread 0 of a K2 CTA) whether this CTA stays for the items past the
// split.  The first K2 CTA to start on an SM decides for the SM: it stays
// if fewer than ovl_stay_sms SMs have been elected.  A later one follows
// that decision; if the decision does not come within the limit, it stays
// (taking more items is always correct).
__device__ bool elect_stay(const ChunkParams& p) {
  uint32_t smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  OverlapCounters* c = p.ovl;
  const uint32_t key = smid % kOvlSmKeys;
  if (atomicAdd(&c->arrived[key], 1u) == 0) {
    const bool stay = atomicAdd(&c->stay_sms, 1u) < (uint32_t)p.ovl_stay_sms;
    st_release_u32(&c->role[key], stay ? 2u : 1u);
    return stay;
  }
  if (!wait_at_least(&c->role[key], 1u, kWaitLimitNs)) return true;
  return ld_acquire_u32(&c->role[key]) == 2u;
}

template <bool kHeadGate, bool kConv>
__global__ void __launch_bounds__(kThreads, 2)
tc_intra_ovl(ChunkParams p, int64_t n_items, const __grid_constant__ RowMaps maps) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ IntraBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ int stay;
  const int tid = threadIdx.x;
  if (tid < 32) tmem_alloc(&tmem_base, 256);
  if (tid == 0) init_intra_bars(&bars);
  // the chunk table, the counters and the flags come from the planning kernel
  pdl_wait();
  if (tid == 0) stay = elect_stay(p) ? 1 : 0;
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // K3 may start once every K2 CTA is running (its CTAs need SMs that
  // leaving K2 CTAs free)
  pdl_launch_dependents();
  intra_items<false, kHeadGate, kConv, true, true>(
      p, maps, IntraPipe{sm, &bars, tmem_base, tid, PipeSync{0}, 0, 0, n_items, stay != 0});
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tmem_base, 256);
}

__global__ void __launch_bounds__(OvlChainCfg::kThreads, 1) tc_inter_ovl(ChunkParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ K3Bars<kOvlNs> bars;
  inter_chain<false, kOvlNs, true, false>(p, (int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z, sm, bars);
  // complete only after K2 (which made every record this chain read): the
  // work after this call on the stream waits for both
  pdl_wait();
}

}  // namespace
}  // namespace tcp

int overlap_chain_columns() { return tcp::kOvlNs; }


cudaError_t launch_tc_overlap(const ChunkParams& p, cudaStream_t stream) {
  using namespace tcp;
  if (!p.rec_ready || !p.ovl || !p.inter || p.ovl_stay_sms < 1 || p.dv % kOvlNs != 0)
    return cudaErrorInvalidValue;
  const bool head = p.gate_per_head != 0, conv = p.conv_width > 0;
  auto k2 = conv ? (head ? tc_intra_ovl<true, true> : tc_intra_ovl<false, true>)
                 : (head ? tc_intra_ovl<true, false> : tc_intra_ovl<false, false>);
  cudaError_t e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem::BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tc_inter_ovl, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)OvlChainCfg::BYTES);
  if (e != cudaSuccess || p.max_chunks == 0 || p.total_tokens == 0) return e;
  RowMaps maps;
  if (!make_row_maps(p, &maps)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t n_items = p.max_chunks * (int64_t)p.H;
  const int64_t grid = n_items < 2 * (int64_t)sms ? n_items : 2 * (int64_t)sms;
  e = launch_maybe_dependent(true, k2, dim3((unsigned)grid), dim3(kThreads), (size_t)Smem::BYTES, stream, p,
                             n_items, maps);
  if (e != cudaSuccess) return e;
  return launch_maybe_dependent(true, tc_inter_ovl,
                                dim3((unsigned)p.num_seqs, (unsigned)p.H, (unsigned)(p.dv / kOvlNs)),
                                dim3(OvlChainCfg::kThreads), (size_t)OvlChainCfg::BYTES, stream, p);
}

}  // namespace kda
