// Placeholder for the tcgen05 path while it is being written.
#include "kda_internal.cuh"
namespace kda {
const bool kHaveTensorCorePath = false;
size_t tc_record_bytes() { return 0; }
cudaError_t launch_tc_prefill(const ChunkParams&, cudaStream_t, cudaEvent_t) { return cudaErrorNotSupported; }
}  // namespace kda
