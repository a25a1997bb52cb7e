// kda_noalloc.cu -- kda_prefill without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they run the prefill: an
// engine that reserves all of HBM for its state pools up front, a plugin
// whose host framework owns every allocation, or a code path where an
// allocation is not permitted because it would synchronise the device.  For
// them kda_prefill_noalloc runs the same kernels as kda_prefill on a
// workspace that lives in a file-scope __device__ array of fixed size,
// kKdaNoAllocScratchBytes, which every GPU that loads this library holds
// until the process exits.
//
// The device address of the array is looked up once per device (the first
// call on that device, with it current); that first call should therefore
// come before any stream capture.  The array is shared by every call: calls
// whose kernels overlap on the GPU race on it.  Nothing in it has to start
// at zero: the planning kernel clears the status word and writes the whole
// chunk table before anything reads them, and every record is written before
// it is read.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kKdaNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kKdaNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

}  // namespace
}  // namespace kda

extern "C" kda_status_t kda_prefill_noalloc(const kda_prefill_args* args, void* stream) {
  using namespace kda;
  const size_t need = kda_prefill_workspace_size(args);
  // invalid arguments: kda_prefill reports why, before any launch
  if (need == 0) return kda_prefill(args, nullptr, 0, stream);
  if (need > kKdaNoAllocScratchBytes) return KDA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
    }
    ptr = g_noalloc_ptr[dev];
  }
  return kda_prefill(args, ptr, kKdaNoAllocScratchBytes, stream);
}
