// kda_tc_intra.cu -- K2, the intra-chunk kernel of the tensor-core prefill:
// persistent, two CTAs of 256 threads per SM, each CTA one item pipeline
// (kda_tc_intra.cuh) walking the (chunk, head) items with stride gridDim.x.
#include "kda_tc_intra.cuh"

namespace kda {
namespace tcp {
namespace {

// TMEM (256 columns) and the mbarriers are set up once per CTA.
template <bool kPoll, bool kHeadGate, bool kConv>
__global__ void __launch_bounds__(kThreads, 2)
tc_intra(ChunkParams p, int64_t n_items, const __grid_constant__ RowMaps maps) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ IntraBars bars;
  __shared__ uint32_t tmem_base;
  if (blockIdx.x >= n_items) return;
  const int tid = threadIdx.x;
  if (tid < 32) tmem_alloc(&tmem_base, 256);
  if (tid == 0) init_intra_bars(&bars);
  // (launched as the planning kernel's programmatic dependent) its chunk
  // table is read from here on; the inter-chunk kernel may then be launched
  // (its CTAs wait for this kernel's completion before they read)
  pdl_wait();
  pdl_launch_dependents();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  intra_items<kPoll, kHeadGate, kConv, false>(
      p, maps, IntraPipe{sm, &bars, tmem_base, tid, PipeSync{0}, (int64_t)blockIdx.x, (int64_t)gridDim.x, n_items});
  fence_before_sync();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tmem_base, 256);
}

}  // namespace

}  // namespace tcp

EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

namespace tcp {

cudaError_t launch_intra(const ChunkParams& p, cudaStream_t stream, bool dependent) {
  const bool head = p.gate_per_head != 0, conv = p.conv_width > 0;
  // (the convolution has no polling instance: its waits keep the suspending
  // form, which honours the limit too, only less promptly)
  const bool poll = p.wait_ns < kPollLimitNs && !conv;
  auto kernel = conv ? (head ? tc_intra<false, true, true> : tc_intra<false, false, true>)
                : poll ? (head ? tc_intra<true, true, false> : tc_intra<true, false, false>)
                       : (head ? tc_intra<false, true, false> : tc_intra<false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Smem::BYTES);
  if (e != cudaSuccess || p.max_chunks == 0 || p.total_tokens == 0) return e;
  RowMaps maps;
  if (!make_row_maps(p, &maps)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t n_items = p.max_chunks * (int64_t)p.H;
  const int64_t grid = n_items < 2 * (int64_t)sms ? n_items : 2 * (int64_t)sms;
  return launch_maybe_dependent(dependent, kernel, dim3((unsigned)grid), dim3(kThreads), (size_t)Smem::BYTES,
                                stream, p, n_items, maps);
}

}  // namespace tcp
}  // namespace kda
