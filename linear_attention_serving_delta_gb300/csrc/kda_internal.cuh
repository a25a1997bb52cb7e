// kda_internal.cuh -- parameter blocks and launcher declarations shared by the
// translation units of libkda (not part of the public ABI).
#pragma once

#include <cuda.h>  // CUtensorMap and the enums of its encoder (fetched at run time)

#include "kda_common.cuh"

namespace kda {

// cuTensorMapEncodeTiled, fetched from the driver once (null if unavailable)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

struct PlanParams {
  int32_t num_seqs;
  int64_t total_tokens;
  const int64_t* cu_seqlens;
  int64_t snapshot_interval;
  const int64_t* boundary_pos;
  const int64_t* cu_boundaries;
  int64_t num_boundaries;
  const int64_t* cu_snapshots;
  int64_t num_snapshots;
  const int32_t* slot_map;  // [map_len] or null: snapshot index -> row of the snapshot buffer
  int64_t map_len;
  int64_t max_chunks;
  // workspace outputs
  int32_t* status;
  PlanMeta* meta;
  int64_t* seq_len;         // [N]
  int64_t* seq_seg_begin;   // [N+1]
  int64_t* seq_chunk_begin; // [N+1]
  int64_t* seq_bnd;         // [2N] usable boundary range per sequence
  int32_t* bnd_nonaligned;  // [num_boundaries + N]
  int32_t* bnd_nonmult;     // [num_boundaries + N]
  Chunk* chunks;            // [max_chunks]
  // (or null) the sequences by chunk count, longest first (ties by index):
  // the inter-chunk kernels start the chains of long sequences first
  int32_t* seq_order;       // [N]
  // words the planning kernel clears before anything else (the overlapped
  // schedule's record flags and counters), or null
  uint32_t* zero_words;
  int64_t n_zero_words;
};

// Counters of the overlapped tensor-core prefill, in the workspace, cleared
// by the planning kernel.  SMs are keyed by their id modulo kOvlSmKeys (two
// SMs that share a key share a role, which changes no result).
constexpr int kOvlSmKeys = 512;
struct OverlapCounters {
  unsigned long long next_item;  // items taken so far
  uint32_t stay_sms;             // SMs elected to stay
  uint32_t pad;
  uint32_t arrived[kOvlSmKeys];  // intra-chunk CTAs started on the SM
  uint32_t role[kOvlSmKeys];     // 0 undecided, 1 leaves at the split, 2 stays
};

// Everything the intra-chunk and inter-chunk kernels read.
struct ChunkParams {
  int32_t num_seqs, H, dk, dv;
  int64_t max_chunks;
  int64_t total_tokens;
  const void* q;
  const void* k;
  const void* v;
  const void* g;
  const void* b;
  float scale;
  const float* initial_state;
  void* o;
  float* final_state;
  float* snapshots;
  // workspace
  int32_t* status;
  const PlanMeta* meta;
  const int64_t* seq_chunk_begin;
  const Chunk* chunks;
  // (or null) the sequences longest first (PlanParams::seq_order): the
  // inter-chunk kernels take their CTAs' sequences in that order, so that
  // the chains that run longest start in the first wave
  const int32_t* seq_order;
  float* inter;     // [max_chunks][H] records
  size_t rec_floats;
  // segment scan (tensor-core path): mode kScanPass1 runs grid z = 0..3 from
  // a zero state (final -> final_state) and z = 4..7 as the transition maps
  // (identity state, U~ taken as zero, final -> trans); no o or snapshots
  int32_t k3_mode;
  float* trans;     // [num_seqs][H][dk][dk] in kScanPass1
  uint64_t wait_ns; // limit of the bounded waits on copies and MMAs (not of the drains)
  int32_t gate_per_head;  // g is [T, H] (one decay per token and head), else [T, H, dk]
  // the layer steps (kda_layer_args): short convolution of q, k, v (width 0 =
  // off) and output gate (null = off)
  int32_t conv_width, conv_silu;
  const float* conv_w[3];   // taps of q, k, v: [conv_width][H][d]
  const void* conv_in[3];   // windows [N][conv_width - 1][H][d], or null (zeros)
  // the chunk table's sequences are segments of the one sequence of the call
  // (segment scan): a chunk's position in it is its first token's index
  int32_t conv_one_seq;
  const void* out_gate;     // [T][H][dv], or [T][H] with out_gate_per_head
  int32_t out_gate_per_head;
  // the fused and the overlapped tensor-core prefill: a flag per record
  // [max_chunks][H], zero at the launch, set once the record is complete
  // (null otherwise)
  uint32_t* rec_ready;
  // the overlapped tensor-core prefill (OverlapCounters, zero at the launch):
  // the intra-chunk CTAs on ovl_stay_sms SMs take items until none is left,
  // the others only while fewer than ovl_split have been taken
  OverlapCounters* ovl;
  int32_t ovl_stay_sms;
  int64_t ovl_split;
};

constexpr int32_t kScanPass1 = 1;

// The window of each sequence after the call (kda_layer_args::conv_out):
// the raw inputs of the last conv_width - 1 positions of window ++ sequence.
// Runs after every kernel that reads conv_in (the two may be one buffer).
cudaError_t launch_conv_windows(const kda_layer_args& l, int32_t num_seqs, int32_t H, int32_t dk,
                                int32_t dv, const int64_t* cu_seqlens, int64_t total_tokens,
                                kda_dtype_t dt, const void* const x[3], cudaStream_t stream);

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);

// A launch as the programmatic dependent of the kernel before it on the
// stream (programmatic stream serialization): its CTAs may start once every
// CTA of that kernel has signalled (pdl_launch_dependents) or exited, and it
// waits for that kernel's results at pdl_wait.  `dependent` false: an
// ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_dependent(bool dependent, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// fp32 CUDA-core path (any supported dk, dv; f32 or bf16 inputs)
// `mid` (may be null) is recorded on the stream between the intra-chunk and
// the inter-chunk kernels.
cudaError_t launch_simt_prefill(const ChunkParams& p, kda_dtype_t dt, cudaStream_t stream,
                                cudaEvent_t mid);

// tcgen05 tensor-core path (bf16 inputs, dk = dv = 128)
extern const bool kHaveTensorCorePath;
size_t tc_record_bytes();
cudaError_t launch_tc_prefill(const ChunkParams& p, cudaStream_t stream, cudaEvent_t mid);
// The fused tensor-core prefill (kda_tc_fused.cu): one launch of `grid`
// CTAs (two per SM), the last n_chain of them the chains of the (sequence,
// head, fused_chain_columns()-column slice) triples in that order, the
// others the intra-chunk item pipelines; p.rec_ready set and zero.
// fused_supported: the device holds two of its CTAs per SM.
int fused_chain_columns();
bool fused_supported(int device);
cudaError_t launch_tc_fused(const ChunkParams& p, int32_t n_chain, int32_t grid, cudaStream_t stream);
// The overlapped tensor-core prefill (kda_tc_overlap.cu): the intra-chunk
// kernel and then the inter-chunk kernel launched as its programmatic
// dependent, the chains starting on the SMs the intra-chunk CTAs leave at
// the split while p.ovl_stay_sms SMs make the last records; p.rec_ready and
// p.ovl set and zero (cleared by the planning kernel launched before).
// overlap_chain_columns: the state columns of a chain CTA.
int overlap_chain_columns();
cudaError_t launch_tc_overlap(const ChunkParams& p, cudaStream_t stream);
// The segment scan over P chunk-aligned segments of one sequence (planned as
// P sequences in `p`): K2 once, K3 pass 1 (state offsets B and transition
// maps A of every segment, in parallel), the combine (inits[s+1] = A_s
// inits[s] + B_s), K3 pass 2 from the true segment states.  Buffers are
// [P][H][128][128] fp32; `s0` may be null (zeros); `final_state` (may be
// null) receives the last segment's final state.
struct ScanBuffers {
  float* A;
  float* B;
  float* inits;
  float* finals;
  const float* s0;
  float* final_state;
};
cudaError_t launch_tc_prefill_scan(const ChunkParams& p, const ScanBuffers& sb, cudaStream_t stream,
                                   cudaEvent_t mid);
// seg_cu[0..P] from cu_seqlens[0..1] of one sequence: chunk-aligned cuts
cudaError_t launch_scan_plan(const int64_t* cu_seqlens, int64_t total_tokens, int32_t P,
                             int64_t* seg_cu, cudaStream_t stream);

cudaError_t launch_decode(const kda_decode_args& a, cudaStream_t stream);
cudaError_t launch_prep(const kda_prep_args& a, cudaStream_t stream);

}  // namespace kda
