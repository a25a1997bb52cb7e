// kda_tc_handoff.cuh -- how the records pass from the item pipelines to the
// chains inside the fused tensor-core prefill.
//
// The fused kernel (kda_tc_fused.cu) runs the intra-chunk step (item
// pipelines, kda_tc_intra.cuh) and the inter-chunk chains (kda_tc_inter.cuh)
// at the same time, on different CTAs.  A pipeline writes the record of
// (chunk cidx, head h) to its place in the record array, as the separate
// intra-chunk kernel does, and then publishes it: p.rec_ready[cidx * H + h]
// (zero at the launch) is set to 1 with release semantics, once the
// record's bulk copies have landed and its plain stores are fenced.  A chain
// copies a record into shared memory only once it sees the flag (acquire,
// then a proxy fence, as the copy is an async-proxy read of data written
// partly through the generic proxy).  The chain follows the pipelines a few
// chunks behind, so it reads each record from L2.
//
// Pipelines never wait for chains, only chains for pipelines, and the
// chains are the last CTAs of the grid: CTAs start in index order, so a
// chain that is running has every pipeline running or done before it, and
// every wait ends.  These waits are for other CTAs' progress, not for a
// copy or an MMA of the waiting CTA: they take the longer of the call's
// wait limit and 1 s.
#pragma once

#include "kda_tc_common.cuh"

namespace kda {
namespace tcp {

using tc::kWaitLimitNs;

__device__ __forceinline__ uint32_t* rec_flag(const ChunkParams& p, int64_t cidx, int h) {
  return p.rec_ready + (size_t)cidx * p.H + h;
}
__device__ __forceinline__ uint64_t handoff_limit_ns(const ChunkParams& p) {
  return p.wait_ns > kWaitLimitNs ? p.wait_ns : kWaitLimitNs;
}

// Record (cidx, h) is complete (the caller has ordered its writes first).
__device__ __forceinline__ void rec_publish(const ChunkParams& p, int64_t cidx, int h) {
  tc::st_release_u32(rec_flag(p, cidx, h), 1u);
}
// Record (cidx, h) is published (no wait).
__device__ __forceinline__ bool rec_published(const ChunkParams& p, int64_t cidx, int h) {
  return tc::ld_acquire_u32(rec_flag(p, cidx, h)) != 0u;
}
// Waits until record (cidx, h) is published; false if the wait gave up.
// The bulk copies that read it are issued after this.
__device__ __forceinline__ bool rec_wait_published(const ChunkParams& p, int64_t cidx, int h) {
  const bool ok = tc::wait_at_least(rec_flag(p, cidx, h), 1u, handoff_limit_ns(p));
  tc::fence_proxy_async_global();
  return ok;
}

}  // namespace tcp
}  // namespace kda
