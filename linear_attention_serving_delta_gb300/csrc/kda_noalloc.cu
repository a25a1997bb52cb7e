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
// In host code the array's name is only a host-side stand-in: its device
// address is looked up with cudaGetSymbolAddress, with the call's device
// current.  The lookup is repeated on every call made outside stream
// capture (so a context that was reset or replaced never sees a stale
// address); a call made while its stream is capturing uses the address its
// device's last uncaptured call found, so the first call on a device must
// come before any stream capture.  The array is shared by every call: calls
// whose kernels overlap on the GPU race on it.  Nothing in it has to start
// at zero: the planning kernel clears the status word and writes the whole
// chunk table before anything reads them, and every record is written before
// it is read.  kda_prefill_noalloc_device_status reads its status word back.
#include <mutex>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kKdaNoAllocScratchBytes = (size_t)64 << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kKdaNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// The array's device address on the current device (see the file comment).
kda_status_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return *out ? KDA_OK : KDA_ERR_CUDA;  // capturing before any uncaptured call
}

}  // namespace
}  // namespace kda

extern "C" kda_status_t kda_prefill_noalloc(const kda_prefill_args* args, void* stream) {
  using namespace kda;
  const size_t need = kda_prefill_workspace_size(args);
  // invalid arguments: kda_prefill reports why, before any launch
  if (need == 0) return kda_prefill(args, nullptr, 0, stream);
  if (need > kKdaNoAllocScratchBytes) return KDA_ERR_WORKSPACE;
  void* ptr = nullptr;
  const kda_status_t st = scratch_address(static_cast<cudaStream_t>(stream), &ptr);
  if (st != KDA_OK) return st;
  return kda_prefill(args, ptr, kKdaNoAllocScratchBytes, stream);
}

extern "C" kda_status_t kda_prefill_noalloc_device_status(int32_t* out, void* stream_) {
  using namespace kda;
  if (!out) return KDA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t v = 0;
  // the status word is the first int32 of the workspace (see kda_prefill_device_status)
  if (cudaMemcpyFromSymbolAsync(&v, g_noalloc_scratch, sizeof(int32_t), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  *out = v;
  return KDA_OK;
}
