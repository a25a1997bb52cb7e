// kda_tc_inter.cu -- K3, the inter-chunk kernel of the tensor-core prefill
// (one chain CTA of kda_tc_inter.cuh per sequence, head and column slice),
// the launcher of the tensor-core prefill (K2 then K3, or the fused kernel
// of kda_tc_fused.cu) and the segment scan's passes.
#include "kda_tc_inter.cuh"

namespace kda {
namespace tcp {
namespace {

template <bool kPoll, int NS>
__global__ void __launch_bounds__(K3Cfg<NS>::kThreads, 1) tc_inter(ChunkParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ K3Bars<NS> bars;
  // (launched as the intra-chunk kernel's programmatic dependent) its
  // records are read from here on
  pdl_wait();
  int s = (int)blockIdx.x, h = (int)blockIdx.y, z = (int)blockIdx.z;
  if (p.seq_order) {
    // CTAs start in the order of their linear index: the sequences longest
    // first, each with all its heads and column slices
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const unsigned per = gridDim.y * gridDim.z, r = lin % per;
    s = p.seq_order[lin / per];
    h = (int)(r / gridDim.z);
    z = (int)(r % gridDim.z);
  }
  inter_chain<kPoll, NS, false>(p, s, h, z, sm, bars);
}

// tc_inter with the wait mode its limit asks for, over grid (gx, gy, zmul x
// the head's column slices)
template <int NS>
cudaError_t run_inter_ns(const ChunkParams& p, unsigned gx, unsigned gy, unsigned zmul, cudaStream_t stream,
                         bool dependent) {
  using C = K3Cfg<NS>;
  const bool poll = p.wait_ns < kPollLimitNs;
  auto kernel = poll ? tc_inter<true, NS> : tc_inter<false, NS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
  if (e != cudaSuccess) return e;
  return launch_maybe_dependent(dependent, kernel, dim3(gx, gy, zmul * (unsigned)(p.dv / NS)), dim3(C::kThreads),
                                (size_t)C::BYTES, stream, p);
}
// 32 state columns per CTA while those CTAs all fit the GPU at once (a chain
// step of a 32-column CTA is shorter), else 64 where the value columns come
// in 64s (half the CTAs, each at a longer step: less time in all once the
// CTAs run in waves)
// dependent: launched as the programmatic dependent of the intra-chunk kernel
cudaError_t run_inter(const ChunkParams& p, unsigned gx, unsigned gy, unsigned zmul, cudaStream_t stream,
                      bool dependent = false) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t ctas32 = (int64_t)gx * gy * zmul * (p.dv / 32);
  return (p.dv % 64 == 0 && ctas32 > sms) ? run_inter_ns<64>(p, gx, gy, zmul, stream, dependent)
                                          : run_inter_ns<32>(p, gx, gy, zmul, stream, dependent);
}

}  // namespace
}  // namespace tcp

const bool kHaveTensorCorePath = true;

size_t tc_record_bytes() { return tcp::Rec::BYTES; }

// The intra-chunk kernel as the planning kernel's programmatic dependent,
// and the inter-chunk kernel as its (unless `mid` sits between them): each
// starts its set-up while the kernel before it finishes.
cudaError_t launch_tc_prefill(const ChunkParams& p, cudaStream_t stream, cudaEvent_t mid) {
  using namespace tcp;
  cudaError_t e = launch_intra(p, stream, true);
  if (e != cudaSuccess) return e;
  if (mid) {
    e = cudaEventRecord(mid, stream);
    if (e != cudaSuccess) return e;
  }
  return run_inter(p, (unsigned)p.num_seqs, (unsigned)p.H, 1, stream, mid == nullptr);
}

namespace {

using namespace tcp;

constexpr int kCombineNs = 32;  // state columns per CTA of the combine

// inits[0] = S0 (or zeros); inits[s+1] = A_s inits[s] + B_s.  One CTA per
// (head, 32-column slice); thread t owns row t / 2 and 16 columns.  The
// slice of the running state sits in shared memory; A_s rows are read
// straight from global memory (L2), 4 floats at a time.
__global__ void __launch_bounds__(256) scan_combine(ScanBuffers sb, int P, int H) {
  __shared__ __align__(16) float S[kD * kCombineNs];
  const int h = blockIdx.x, n0 = blockIdx.y * kCombineNs;
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 16;
  const size_t mat = (size_t)kD * kD;
  float acc[16];
  {
    const float* s0 = sb.s0 ? sb.s0 + (size_t)h * mat + (size_t)r * kD + n0 + c0 : nullptr;
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n] = s0 ? s0[n] : 0.f;
  }
  for (int s = 0;; ++s) {
    float* out = sb.inits + ((size_t)s * H + h) * mat + (size_t)r * kD + n0 + c0;
#pragma unroll
    for (int n = 0; n < 16; n += 4) {
      *reinterpret_cast<float4*>(out + n) = make_float4(acc[n], acc[n + 1], acc[n + 2], acc[n + 3]);
      *reinterpret_cast<float4*>(S + r * kCombineNs + c0 + n) = make_float4(acc[n], acc[n + 1], acc[n + 2], acc[n + 3]);
    }
    if (s + 1 >= P) break;
    __syncthreads();
    const float* a = sb.A + ((size_t)s * H + h) * mat + (size_t)r * kD;
    const float* b = sb.B + ((size_t)s * H + h) * mat + (size_t)r * kD + n0 + c0;
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n] = b[n];
    for (int k = 0; k < kD; k += 4) {
      const float4 a4 = __ldg(reinterpret_cast<const float4*>(a + k));
      const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float* srow = S + (k + kk) * kCombineNs + c0;
#pragma unroll
        for (int n = 0; n < 16; n += 4) {
          const float4 x = *reinterpret_cast<const float4*>(srow + n);
          acc[n] += av[kk] * x.x;
          acc[n + 1] += av[kk] * x.y;
          acc[n + 2] += av[kk] * x.z;
          acc[n + 3] += av[kk] * x.w;
        }
      }
    }
    __syncthreads();  // every row of S read before it is overwritten
  }
}

// Chunk-aligned cuts of one sequence [cu[0], cu[1]) into P segments.  A
// malformed cu (cu[0] != 0, or cu[1] outside [0, total_tokens]) yields
// segments the planning kernel flags (start 1) and skips (all empty).
__global__ void scan_plan(const int64_t* cu, int64_t total_tokens, int32_t P, int64_t* seg_cu) {
  if (threadIdx.x != 0) return;
  const int64_t c0 = cu[0], len = cu[1] - cu[0];
  if (c0 != 0 || len < 0 || cu[1] > total_tokens) {
    for (int32_t s = 0; s <= P; ++s) seg_cu[s] = 1;
    return;
  }
  const int64_t nch = (len + kChunk - 1) / kChunk;
  const int64_t step = ((nch + P - 1) / P) * kChunk;
  for (int32_t s = 0; s <= P; ++s) seg_cu[s] = s * step < len ? s * step : len;
}

}  // namespace

cudaError_t launch_scan_plan(const int64_t* cu_seqlens, int64_t total_tokens, int32_t P,
                             int64_t* seg_cu, cudaStream_t stream) {
  scan_plan<<<1, 32, 0, stream>>>(cu_seqlens, total_tokens, P, seg_cu);
  return cudaGetLastError();
}

cudaError_t launch_tc_prefill_scan(const ChunkParams& p, const ScanBuffers& sb, cudaStream_t stream,
                                   cudaEvent_t mid) {
  using namespace tcp;
  cudaError_t e = launch_intra(p, stream);
  if (e != cudaSuccess) return e;
  if (mid) {
    e = cudaEventRecord(mid, stream);
    if (e != cudaSuccess) return e;
  }
  // pass 1: the state offset B_s and the transition map A_s of every segment
  ChunkParams p1 = p;
  p1.k3_mode = kScanPass1;
  p1.initial_state = nullptr;
  p1.final_state = sb.B;
  p1.trans = sb.A;
  p1.snapshots = nullptr;
  e = run_inter(p1, (unsigned)p.num_seqs, (unsigned)p.H, 2, stream);
  if (e != cudaSuccess) return e;
  scan_combine<<<dim3((unsigned)p.H, (unsigned)(kD / kCombineNs)), 256, 0, stream>>>(sb, p.num_seqs, p.H);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // pass 2: every segment from its true initial state
  ChunkParams p2 = p;
  p2.k3_mode = 0;
  p2.initial_state = sb.inits;
  p2.final_state = sb.finals;
  p2.trans = nullptr;
  e = run_inter(p2, (unsigned)p.num_seqs, (unsigned)p.H, 1, stream);
  if (e != cudaSuccess || !sb.final_state) return e;
  return cudaMemcpyAsync(sb.final_state, sb.finals + (size_t)(p.num_seqs - 1) * p.H * kD * kD,
                         (size_t)p.H * kD * kD * sizeof(float), cudaMemcpyDeviceToDevice, stream);
}

}  // namespace kda
