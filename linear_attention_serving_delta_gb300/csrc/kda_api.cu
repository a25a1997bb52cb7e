// kda_api.cu -- the extern "C" entry points of libkda: argument validation,
// workspace layout and kernel launches.  Declarations and contracts are in
// include/kda.h.
#include <new>

#include "kda_internal.cuh"

namespace kda {
namespace {

bool head_size_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }
bool dtype_ok(kda_dtype_t t) { return t == KDA_F32 || t == KDA_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The layer steps' buffers read with 16-byte vector accesses on the
// tensor-core path (taps, windows, a per-channel output gate).
bool layer_aligned16(const kda_layer_args* l) {
  if (!l) return true;
  for (int t = 0; t < 3; ++t)
    if (l->conv_width > 0 && (!aligned16(l->conv_w[t]) || !aligned16(l->conv_in[t]))) return false;
  return l->out_gate_per_head || aligned16(l->out_gate);
}

// The tensor-core kernels move q, k, g, v, o and the states with 16-byte
// vector accesses; other layouts take the fp32 CUDA-core path.
// The tensor-core path: bf16, heads of up to 128 channels (a narrower head
// runs zero-padded to 128: its tensor-map copies fill the missing channels
// with zeros, which changes no product, and the outputs keep the caller's
// layout; dv a multiple of the inter-chunk kernel's 32-column slice),
// 16-byte aligned buffers, and token indices that fit the int32 coordinates
// of its tensor-map copies.  The short convolution's staging is laid out for
// 128 channels: with it, only 128 x 128 heads.
bool use_tensor_cores(const kda_prefill_args* a) {
  const bool conv = a->layer && a->layer->conv_width > 0;
  return kHaveTensorCorePath && a->in_dtype == KDA_BF16 && a->dk <= 128 && a->dv >= 32 && a->dv <= 128 &&
         (!conv || (a->dk == 128 && a->dv == 128)) && a->total_tokens < ((int64_t)1 << 31) &&
         aligned16(a->q) && aligned16(a->k) && aligned16(a->v) && aligned16(a->g) &&
         aligned16(a->o) && aligned16(a->initial_state) && aligned16(a->final_state) &&
         aligned16(a->snapshots) && layer_aligned16(a->layer);
}

// Byte ranges [p, p + n) that overlap without being the same range.
bool partly_overlap(const void* p, const void* q, size_t n) {
  if (!p || !q || p == q) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + n && b < a + n;
}

// The layer steps' arguments (kda.h): `rows` = sequences (prefill) or state
// slots (decode); `elem` = bytes per element of in_dtype.
kda_status_t validate_layer(const kda_layer_args* l, int64_t rows, int32_t H, int32_t dk, int32_t dv,
                            size_t elem) {
  if (!l) return KDA_OK;
  if (l->conv_width < 0 || l->conv_width > KDA_CONV_MAX) return KDA_ERR_INVALID_ARG;
  if (l->out_gate_per_head != 0 && l->out_gate_per_head != 1) return KDA_ERR_INVALID_ARG;
  if (l->conv_width > 0) {
    const int32_t d[3] = {dk, dk, dv};
    for (int t = 0; t < 3; ++t) {
      if (!l->conv_w[t]) return KDA_ERR_INVALID_ARG;
      const size_t bytes = (size_t)rows * (l->conv_width - 1) * H * d[t] * elem;
      if (partly_overlap(l->conv_in[t], l->conv_out[t], bytes)) return KDA_ERR_INVALID_ARG;
    }
  }
  return KDA_OK;
}

size_t elem_bytes(kda_dtype_t t) { return t == KDA_BF16 ? 2 : 4; }

constexpr int32_t kMaxScanSegments = 64;
constexpr int32_t kScanSms = 152;  // SMs of the part the automatic choice is sized for

// Segments of the segment scan for these arguments (host-side fields only):
// 1 = no scan.  See kda.h.
int32_t scan_segments_of(const kda_prefill_args* a) {
  if (!use_tensor_cores(a) || a->dk != 128 || a->dv != 128 || a->num_seqs != 1 ||
      a->snapshot_interval != 0 || a->boundary_pos ||
      a->snapshots || a->scan_segments == 1)
    return 1;
  const int64_t nch = (a->total_tokens + kChunk - 1) / kChunk;
  int64_t P;
  if (a->scan_segments >= 2) {
    P = a->scan_segments;
  } else {
    P = kScanSms / (8 * (int64_t)a->num_heads);
    if (nch / 16 < P) P = nch / 16;
    if (P < 3) return 1;
  }
  return (int32_t)(P > kMaxScanSegments ? kMaxScanSegments : P);
}

kda_status_t validate_prefill(const kda_prefill_args* a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->num_seqs < 1 || a->num_heads < 1 || a->total_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype)) return KDA_ERR_INVALID_ARG;
  if (!head_size_ok(a->dk) || !head_size_ok(a->dv)) return KDA_ERR_UNSUPPORTED;
  if (!a->cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->g || !a->b || !a->o))
    return KDA_ERR_INVALID_ARG;
  if (a->snapshot_interval < 0 || a->snapshot_interval % KDA_CHUNK != 0) return KDA_ERR_INVALID_ARG;
  if ((a->boundary_pos == nullptr) != (a->cu_boundaries == nullptr)) return KDA_ERR_INVALID_ARG;
  if (a->num_boundaries < 0 || (!a->boundary_pos && a->num_boundaries != 0))
    return KDA_ERR_INVALID_ARG;
  if ((a->snapshots == nullptr) != (a->cu_snapshots == nullptr)) return KDA_ERR_INVALID_ARG;
  if (a->num_snapshots < 0 || (a->snapshots && a->num_snapshots == 0)) return KDA_ERR_INVALID_ARG;
  if (a->scan_segments < 0 || a->scan_segments > kMaxScanSegments) return KDA_ERR_INVALID_ARG;
  if (a->snapshot_slot_map && (!a->snapshots || a->snapshot_map_len < 0)) return KDA_ERR_INVALID_ARG;
  if (!a->snapshot_slot_map && a->snapshot_map_len != 0) return KDA_ERR_INVALID_ARG;
  if (a->wait_limit_ns < 0) return KDA_ERR_INVALID_ARG;
  if (a->gate_per_head != 0 && a->gate_per_head != 1) return KDA_ERR_INVALID_ARG;
  if (a->schedule != KDA_SCHEDULE_AUTO && a->schedule != KDA_SCHEDULE_SEPARATE &&
      a->schedule != KDA_SCHEDULE_FUSED && a->schedule != KDA_SCHEDULE_OVERLAP)
    return KDA_ERR_INVALID_ARG;
  kda_status_t ls = validate_layer(a->layer, a->num_seqs, a->num_heads, a->dk, a->dv, elem_bytes(a->in_dtype));
  if (ls != KDA_OK) return ls;
  // sizes whose products must stay inside the index types used by the kernels
  if (a->total_tokens > ((int64_t)1 << 40)) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

// The fused tensor-core prefill applies to these arguments when its chains
// (one per sequence, head and 32-column slice) are at most as many as the
// SMs: each takes half an SM beside an item CTA.  Host-side fields only, and
// the SM count.
bool fused_shape(const kda_prefill_args* a) {
  return use_tensor_cores(a) && scan_segments_of(a) == 1 && a->dv % fused_chain_columns() == 0 &&
         a->total_tokens > 0;
}
int64_t fused_chains(const kda_prefill_args* a) {
  return (int64_t)a->num_seqs * a->num_heads * (a->dv / fused_chain_columns());
}
bool fused_fits(const kda_prefill_args* a, int sms) {
  return a->schedule == KDA_SCHEDULE_FUSED && fused_shape(a) && fused_chains(a) <= sms;
}

// The overlapped tensor-core prefill (kda_tc_overlap.cu) applies to one
// sequence without the segment scan, with normal wait limits (the give-up
// test's short limits take the separate kernels).  Host-side fields only.
bool overlap_shape(const kda_prefill_args* a) {
  return use_tensor_cores(a) && scan_segments_of(a) == 1 && a->num_seqs == 1 && a->dv % 32 == 0 &&
         a->total_tokens > 0 && (a->wait_limit_ns == 0 || a->wait_limit_ns >= 100000) &&
         (a->schedule == KDA_SCHEDULE_AUTO || a->schedule == KDA_SCHEDULE_OVERLAP);
}
int64_t overlap_chains(const kda_prefill_args* a) {
  return (int64_t)a->num_seqs * a->num_heads * (a->dv / 32);
}
// Where it is taken on a GPU of `sms` SMs: its chains (one per head and
// 32-column slice of the state, an SM each) take at most half the SMs, so
// that the SMs left to the intra-chunk kernel make the last records about as
// fast as the chains read them; the automatic choice also wants at least
// kOvlMinChains of them.  Measured on GB300 (one sequence, bf16, L2
// flushed): 64 chains (32 heads of 64 channels, 16 heads of 128, 8192 and
// 65536 tokens) 1.12-1.21x the separate kernels; 32 chains 0.99-1.0x;
// 96 and 128 chains 0.93-0.99x (24-56 SMs left make the last records too
// slowly).
constexpr int64_t kOvlMinChains = 40;
bool overlap_fits(const kda_prefill_args* a, int sms) {
  const int64_t n = overlap_chains(a);
  return overlap_shape(a) && 2 * n <= sms && (a->schedule == KDA_SCHEDULE_OVERLAP || n >= kOvlMinChains);
}

// The split of the overlapped prefill: the intra-chunk CTAs that leave stop
// taking items once this many are taken.  The staying SMs (2 CTAs each) then
// make the remaining items while the chains run.  A chain step takes about
// kOvlStepPerItem of an intra-chunk item's time in one CTA (measured on
// GB300: 12.2 us an item at two CTAs per SM, 1.44 us a chain step), so R
// remaining items keep ahead of the chains when R <= 2 stay x chunks x
// kOvlStepPerItem; a margin below that.
constexpr double kOvlStepPerItem = 0.118;
constexpr double kOvlMargin = 0.85;
int64_t overlap_split(const kda_prefill_args* a, int32_t stay_sms) {
  const int64_t chunks = (a->total_tokens + kChunk - 1) / kChunk + a->num_boundaries;
  const double ratio = kOvlStepPerItem * kOvlMargin;
  const int64_t rest = (int64_t)(ratio * 2.0 * stay_sms * (double)chunks);
  const int64_t items = chunks * a->num_heads;
  return items > rest ? items - rest : 0;
}

WsLayout prefill_layout(const kda_prefill_args* a) {
  WsLayout L;
  // with the segment scan the planner sees P sequences (the segments)
  const int32_t P = scan_segments_of(a);
  const int64_t N = P > 1 ? P : a->num_seqs, nb = a->num_boundaries;
  L.max_chunks = (a->total_tokens + kChunk - 1) / kChunk + N + nb;
  L.rec_bytes = use_tensor_cores(a) ? tc_record_bytes()
                                    : SimtRec::floats(a->dk, a->dv) * sizeof(float);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.status = take(sizeof(int32_t) * 4);
  L.meta = take(sizeof(PlanMeta));
  L.seq_len = 0;
  L.seq_seg_begin = take(sizeof(int64_t) * (N + 1));
  L.seq_chunk_begin = take(sizeof(int64_t) * (N + 1));
  L.bnd_nonaligned = take(sizeof(int32_t) * (nb + N + 1));
  L.bnd_nonmult = take(sizeof(int32_t) * (nb + N + 1));
  L.seq_aux = take(sizeof(int64_t) * 3 * N);  // seq_len [N] + seq_bnd [2N]
  L.seq_order = take(sizeof(int32_t) * N);
  L.chunks = take(sizeof(Chunk) * (size_t)L.max_chunks);
  L.inter = take(L.rec_bytes * (size_t)L.max_chunks * (size_t)a->num_heads);
  if (fused_shape(a) && a->schedule == KDA_SCHEDULE_FUSED)
    L.rec_ready = take(sizeof(uint32_t) * (size_t)L.max_chunks * a->num_heads);
  if (overlap_shape(a)) {
    // the counters, then the record flags: one region the planning kernel
    // clears (a multiple of 16 bytes)
    L.ovl = take(sizeof(OverlapCounters));
    L.rec_ready = take(sizeof(uint32_t) * (size_t)L.max_chunks * a->num_heads);
    L.ovl_words = (off - L.ovl) / sizeof(uint32_t);
  }
  L.scan_P = P;
  if (P > 1) {
    const size_t mats = (size_t)P * a->num_heads * a->dk * a->dv * sizeof(float);
    L.scan_cu = take(sizeof(int64_t) * (P + 1));
    L.scan_A = take(mats);
    L.scan_B = take(mats);
    L.scan_inits = take(mats);
    L.scan_finals = take(mats);
  }
  L.total = off;
  return L;
}

kda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_prefill_workspace_size(const kda_prefill_args* args) {
  if (validate_prefill(args) != KDA_OK) return 0;
  return prefill_layout(args).total;
}

int32_t kda_prefill_schedule(const kda_prefill_args* a, int32_t sm_count) {
  if (validate_prefill(a) != KDA_OK || sm_count < 0) return -1;
  if (!use_tensor_cores(a)) return KDA_PATH_CUDA_CORES;
  if (scan_segments_of(a) > 1) return KDA_PATH_SEGMENT_SCAN;
  bool device_ok = true;
  if (sm_count == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return -1;
    device_ok = fused_supported(dev);
  }
  if (overlap_fits(a, sm_count)) return KDA_PATH_OVERLAP;
  return device_ok && fused_fits(a, sm_count) ? KDA_PATH_FUSED : KDA_PATH_SEPARATE;
}

kda_status_t kda_prefill(const kda_prefill_args* a, void* ws, size_t ws_bytes, void* stream_) {
  kda_status_t st = validate_prefill(a);
  if (st != KDA_OK) return st;
  const WsLayout L = prefill_layout(a);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return KDA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  char* w = static_cast<char*>(ws);

  const int32_t P = L.scan_P;
  PlanParams pp{};
  pp.num_seqs = P > 1 ? P : a->num_seqs;
  pp.total_tokens = a->total_tokens;
  pp.cu_seqlens = P > 1 ? reinterpret_cast<const int64_t*>(w + L.scan_cu) : a->cu_seqlens;
  pp.snapshot_interval = a->snapshot_interval;
  pp.boundary_pos = a->boundary_pos;
  pp.cu_boundaries = a->cu_boundaries;
  pp.num_boundaries = a->num_boundaries;
  pp.cu_snapshots = a->cu_snapshots;
  pp.num_snapshots = a->snapshots ? a->num_snapshots : 0;
  pp.slot_map = a->snapshot_slot_map;
  pp.map_len = a->snapshot_slot_map ? a->snapshot_map_len : 0;
  pp.max_chunks = L.max_chunks;
  pp.status = reinterpret_cast<int32_t*>(w + L.status);
  pp.meta = reinterpret_cast<PlanMeta*>(w + L.meta);
  pp.seq_seg_begin = reinterpret_cast<int64_t*>(w + L.seq_seg_begin);
  pp.seq_chunk_begin = reinterpret_cast<int64_t*>(w + L.seq_chunk_begin);
  pp.bnd_nonaligned = reinterpret_cast<int32_t*>(w + L.bnd_nonaligned);
  pp.bnd_nonmult = reinterpret_cast<int32_t*>(w + L.bnd_nonmult);
  pp.seq_len = reinterpret_cast<int64_t*>(w + L.seq_aux);
  pp.seq_bnd = pp.seq_len + a->num_seqs;
  // the chains of long sequences first, where several sequences' chains
  // share the GPU (the plain tensor-core and CUDA-core prefill)
  if (P == 1 && a->num_seqs > 1) pp.seq_order = reinterpret_cast<int32_t*>(w + L.seq_order);
  pp.chunks = reinterpret_cast<Chunk*>(w + L.chunks);

  // the path on the tensor cores (no device query for the other paths)
  int dev = 0, sms = 0;
  bool overlap = false;
  if (P == 1 && use_tensor_cores(a)) {
    cudaError_t qe = cudaGetDevice(&dev);
    if (qe == cudaSuccess) qe = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (qe != cudaSuccess) return KDA_ERR_CUDA;
    overlap = overlap_fits(a, sms);
  }
  if (overlap) {
    pp.zero_words = reinterpret_cast<uint32_t*>(w + L.ovl);
    pp.n_zero_words = L.ovl_words;
  }

  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->phase_events);
  auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], stream) : cudaSuccess; };

  cudaError_t e = mark(0);
  if (e == cudaSuccess && P > 1)
    e = launch_scan_plan(a->cu_seqlens, a->total_tokens, P, reinterpret_cast<int64_t*>(w + L.scan_cu),
                         stream);
  if (e == cudaSuccess) e = launch_plan(pp, stream);
  if (e == cudaSuccess) e = mark(1);
  if (e != cudaSuccess) return KDA_ERR_CUDA;

  ChunkParams cp{};
  cp.num_seqs = pp.num_seqs;
  cp.H = a->num_heads;
  cp.dk = a->dk;
  cp.dv = a->dv;
  cp.max_chunks = L.max_chunks;
  cp.total_tokens = a->total_tokens;
  cp.q = a->q;
  cp.k = a->k;
  cp.v = a->v;
  cp.g = a->g;
  cp.b = a->b;
  cp.scale = a->scale;
  cp.initial_state = a->initial_state;
  cp.o = a->o;
  cp.final_state = a->final_state;
  cp.snapshots = a->snapshots;
  cp.status = pp.status;
  cp.meta = pp.meta;
  cp.seq_chunk_begin = pp.seq_chunk_begin;
  cp.seq_order = pp.seq_order;
  cp.chunks = pp.chunks;
  cp.inter = reinterpret_cast<float*>(w + L.inter);
  cp.rec_floats = L.rec_bytes / sizeof(float);
  cp.wait_ns = a->wait_limit_ns > 0 ? (uint64_t)a->wait_limit_ns : 1000000000ull;
  cp.gate_per_head = a->gate_per_head;
  if (const kda_layer_args* l = a->layer) {
    cp.conv_width = l->conv_width;
    cp.conv_silu = l->conv_silu != 0;
    for (int t = 0; t < 3; ++t) {
      cp.conv_w[t] = l->conv_width > 0 ? l->conv_w[t] : nullptr;
      cp.conv_in[t] = l->conv_width > 1 ? l->conv_in[t] : nullptr;
    }
    cp.conv_one_seq = P > 1;
    cp.out_gate = l->out_gate;
    cp.out_gate_per_head = l->out_gate_per_head;
  }
  if (P > 1) {
    ScanBuffers sb;
    sb.A = reinterpret_cast<float*>(w + L.scan_A);
    sb.B = reinterpret_cast<float*>(w + L.scan_B);
    sb.inits = reinterpret_cast<float*>(w + L.scan_inits);
    sb.finals = reinterpret_cast<float*>(w + L.scan_finals);
    sb.s0 = a->initial_state;
    sb.final_state = a->final_state;
    e = launch_tc_prefill_scan(cp, sb, stream, ev ? ev[2] : nullptr);
  } else if (overlap) {
    cp.rec_ready = reinterpret_cast<uint32_t*>(w + L.rec_ready);
    cp.ovl = reinterpret_cast<OverlapCounters*>(w + L.ovl);
    cp.ovl_stay_sms = sms - (int32_t)overlap_chains(a);
    cp.ovl_split = overlap_split(a, cp.ovl_stay_sms);
    e = launch_tc_overlap(cp, stream);
    if (e == cudaSuccess && ev) e = cudaEventRecord(ev[2], stream);
  } else if (use_tensor_cores(a)) {
    if (fused_fits(a, sms) && fused_supported(dev)) {
      cp.rec_ready = reinterpret_cast<uint32_t*>(w + L.rec_ready);
      e = cudaMemsetAsync(cp.rec_ready, 0, sizeof(uint32_t) * (size_t)L.max_chunks * a->num_heads, stream);
      if (e == cudaSuccess) e = launch_tc_fused(cp, (int32_t)fused_chains(a), 2 * sms, stream);
      if (e == cudaSuccess && ev) e = cudaEventRecord(ev[2], stream);
    } else {
      e = launch_tc_prefill(cp, stream, ev ? ev[2] : nullptr);
    }
  } else {
    e = launch_simt_prefill(cp, a->in_dtype, stream, ev ? ev[2] : nullptr);
  }
  if (e == cudaSuccess && a->layer && a->layer->conv_width > 1) {
    const void* x[3] = {a->q, a->k, a->v};
    e = launch_conv_windows(*a->layer, a->num_seqs, a->num_heads, a->dk, a->dv, a->cu_seqlens,
                            a->total_tokens, a->in_dtype, x, stream);
  }
  if (e == cudaSuccess) e = mark(3);
  return from_cuda(e);
}

kda_status_t kda_prefill_device_status(const void* ws, int32_t* out, void* stream_) {
  if (!ws || !out) return KDA_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return KDA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  *out = v;
  return KDA_OK;
}

int64_t kda_snapshot_plan(const int64_t* h_cu, int32_t n, int64_t interval,
                          const int64_t* h_bpos, const int64_t* h_cub, int64_t* out) {
  if (!h_cu || !out || n < 1 || interval < 0) return -1;
  if ((h_bpos == nullptr) != (h_cub == nullptr)) return -1;
  out[0] = 0;
  for (int32_t s = 0; s < n; ++s) {
    const int64_t len = h_cu[s + 1] - h_cu[s];
    if (len < 0) return -1;
    int64_t cnt = interval > 0 ? len / interval : 0;
    if (h_bpos) {
      for (int64_t i = h_cub[s]; i < h_cub[s + 1]; ++i) {
        const int64_t x = h_bpos[i];
        if (x < 1 || x > len || (i > h_cub[s] && x <= h_bpos[i - 1])) return -1;
        if (interval <= 0 || x % interval != 0) ++cnt;
      }
    }
    out[s + 1] = out[s] + cnt;
  }
  return out[n];
}

kda_status_t kda_decode_step(const kda_decode_args* a, void* stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->num_heads < 1 || a->num_slots < 0) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype)) return KDA_ERR_INVALID_ARG;
  if (!head_size_ok(a->dk) || !head_size_ok(a->dv)) return KDA_ERR_UNSUPPORTED;
  if (a->batch == 0) return KDA_OK;
  if (!a->q || !a->k || !a->v || !a->g || !a->b || !a->state || !a->o) return KDA_ERR_INVALID_ARG;
  if (!a->state_slots && a->num_slots < a->batch) return KDA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->state) & 15) != 0) return KDA_ERR_INVALID_ARG;
  if (a->wait_limit_ns < 0) return KDA_ERR_INVALID_ARG;
  if (a->gate_per_head != 0 && a->gate_per_head != 1) return KDA_ERR_INVALID_ARG;
  kda_status_t ls = validate_layer(a->layer, a->num_slots, a->num_heads, a->dk, a->dv, elem_bytes(a->in_dtype));
  if (ls != KDA_OK) return ls;
  // heads wider than 128 x 128 run as several CTAs per (row, head), which
  // would race on a q/k window updated in place
  if (a->layer && a->layer->conv_width > 0 && (int64_t)a->dk * a->dv > 128 * 128) return KDA_ERR_UNSUPPORTED;
  return from_cuda(launch_decode(*a, static_cast<cudaStream_t>(stream)));
}

kda_status_t kda_prep(const kda_prep_args* a, void* stream) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->num_seqs < 1 || a->num_heads < 1 || a->total_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (!dtype_ok(a->in_dtype)) return KDA_ERR_INVALID_ARG;
  if (!head_size_ok(a->dk)) return KDA_ERR_UNSUPPORTED;
  if (!a->cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (a->total_tokens > 0 &&
      (!a->q || !a->k || !a->g || !a->b || !a->qhat || !a->khat || !a->G || !a->beta))
    return KDA_ERR_INVALID_ARG;
  if (a->gate_per_head != 0 && a->gate_per_head != 1) return KDA_ERR_INVALID_ARG;
  if (const kda_layer_args* l = a->layer) {
    if (l->conv_width < 0 || l->conv_width > KDA_CONV_MAX) return KDA_ERR_INVALID_ARG;
    if (l->conv_width > 0 && (!l->conv_w[0] || !l->conv_w[1])) return KDA_ERR_INVALID_ARG;
  }
  return from_cuda(launch_prep(*a, static_cast<cudaStream_t>(stream)));
}

const char* kda_status_string(kda_status_t s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported head size or dtype";
    case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case KDA_ERR_CUDA: return "CUDA launch or query failed";
    case KDA_ERR_TIMEOUT: return "bounded device wait expired";
    case KDA_ERR_DEVICE_DATA: return "malformed device-side index data";
  }
  return "unknown status";
}

const char* kda_version(void) { return "libkda 0.1 (sm_103a)"; }

}  // extern "C"
