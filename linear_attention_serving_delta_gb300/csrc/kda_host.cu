// kda_host.cu -- kda_prefill_host: the prefill from host buffers, with the
// host<->device copies of one piece of the batch overlapping the prefill of
// another.  Contract in include/kda.h.
//
// The link between host and device memory moves about 210 GB/s one way and
// 340 GB/s both ways at once on this part, against ~6.8 TB/s of HBM: copying
// a prompt's q, k, v, g, b in takes several times longer than its prefill.
// Cutting the batch into pieces lets the copy engines run back to back while
// the kernels of an earlier piece run; the host work per piece is a few
// asynchronous calls, so many pieces cost little.
#include <vector>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMaxSegments = 64;

struct Piece {
  int64_t tok0, tok1;  // packed token range
  int32_t seq0, nseq;  // sequences [seq0, seq0 + nseq)
  bool split;          // part of one sequence cut at chunk boundaries
  int64_t cu_off;      // entries into the device table of per-piece cu_seqlens
};

bool head_ok(int32_t d) { return d == 16 || d == 32 || d == 64 || d == 128 || d == 256; }

kda_status_t validate_host(const kda_prefill_host_args* a) {
  if (!a) return KDA_ERR_INVALID_ARG;
  if (a->num_seqs < 1 || a->num_heads < 1 || a->total_tokens < 0) return KDA_ERR_INVALID_ARG;
  if (a->in_dtype != KDA_F32 && a->in_dtype != KDA_BF16) return KDA_ERR_INVALID_ARG;
  if (!head_ok(a->dk) || !head_ok(a->dv)) return KDA_ERR_UNSUPPORTED;
  if (!a->cu_seqlens) return KDA_ERR_INVALID_ARG;
  if (a->total_tokens > 0 && (!a->q || !a->k || !a->v || !a->g || !a->b || !a->o))
    return KDA_ERR_INVALID_ARG;
  if (a->segments < 0 || a->segments > kMaxSegments) return KDA_ERR_INVALID_ARG;
  if (a->gate_per_head != 0 && a->gate_per_head != 1) return KDA_ERR_INVALID_ARG;
  if (a->total_tokens > ((int64_t)1 << 40)) return KDA_ERR_UNSUPPORTED;
  const int64_t* cu = a->cu_seqlens;
  if (cu[0] != 0 || cu[a->num_seqs] != a->total_tokens) return KDA_ERR_INVALID_ARG;
  for (int32_t s = 0; s < a->num_seqs; ++s)
    if (cu[s + 1] < cu[s]) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

// The pieces of the pipeline (host-side fields only).
std::vector<Piece> plan_pieces(const kda_prefill_host_args* a) {
  const int64_t T = a->total_tokens, N = a->num_seqs;
  const int64_t nchunks = (T + KDA_CHUNK - 1) / KDA_CHUNK;
  // default: one piece per 48 chunks, at most 4 (each piece costs the copy
  // engines a few microseconds per tensor; the halving tail below already
  // keeps the unoverlapped end short)
  int64_t want = a->segments > 0 ? a->segments : nchunks / 48;
  want = want < 1 ? 1 : (want > 4 && a->segments == 0 ? 4 : want);
  std::vector<Piece> pieces;
  if (N == 1) {
    // chunk-aligned cuts of the one sequence: pieces of about nchunks / want
    // chunks, except that the end is cut into halving pieces (U/8, U/4, U/2
    // chunks): nothing overlaps the prefill and the copy-out of the last
    // piece, so it is kept short
    std::vector<int64_t> sizes;  // in chunks, from the end backwards
    if (want <= 1 || nchunks <= 1) {
      sizes.push_back(nchunks);
    } else {
      const int64_t U = (nchunks + want - 1) / want;
      int64_t left = nchunks, sz = U / 8 > 0 ? U / 8 : 1;
      while (left > 0) {
        const int64_t take = sz < left ? sz : left;
        sizes.push_back(take);
        left -= take;
        sz = 2 * sz < U ? 2 * sz : U;
      }
    }
    int64_t t0 = 0;
    for (size_t i = sizes.size(); i-- > 0;) {
      const int64_t t1 = t0 + sizes[i] * KDA_CHUNK < T ? t0 + sizes[i] * KDA_CHUNK : T;
      pieces.push_back({t0, t1, 0, 1, sizes.size() > 1, 0});
      t0 = t1;
    }
  } else {
    // whole sequences, a new piece once about T / want tokens are gathered
    const int64_t* cu = a->cu_seqlens;
    const int64_t target = T > want ? (T + want - 1) / want : 1;
    int32_t s0 = 0;
    for (int32_t s = 0; s < N; ++s) {
      const bool last = s + 1 == N;
      if (last || cu[s + 1] - cu[s0] >= target) {
        pieces.push_back({cu[s0], cu[s + 1], s0, s + 1 - s0, false, 0});
        s0 = s + 1;
      }
    }
  }
  int64_t off = 0;
  for (Piece& p : pieces) {
    p.cu_off = off;
    off += p.nseq + 1;
  }
  return pieces;
}

struct HostLayout {
  size_t pws, pws_bytes;             // kda_prefill workspace (first, so its status word is ws's)
  size_t q, k, v, g, b, o;           // device copies of the token tensors
  size_t init, fin, carry;           // states: initial, final, two carried between pieces
  size_t cu_all, cu_piece, acc;      // cu_seqlens, per-piece cu tables, status accumulator
  size_t total;
};

// kda_prefill_args of one piece over device copies based at `w`
kda_prefill_args piece_args(const kda_prefill_host_args* a, const HostLayout& L, char* w,
                            const std::vector<Piece>& pieces, size_t i) {
  const Piece& p = pieces[i];
  const int64_t H = a->num_heads, es = a->in_dtype == KDA_BF16 ? 2 : 4;
  const int64_t state = H * a->dk * a->dv;
  kda_prefill_args s{};
  s.num_seqs = p.nseq;
  s.num_heads = a->num_heads;
  s.dk = a->dk;
  s.dv = a->dv;
  s.total_tokens = p.tok1 - p.tok0;
  s.cu_seqlens = reinterpret_cast<const int64_t*>(w + L.cu_piece) + p.cu_off;
  s.in_dtype = a->in_dtype;
  s.q = w + L.q + p.tok0 * H * a->dk * es;
  s.k = w + L.k + p.tok0 * H * a->dk * es;
  s.v = w + L.v + p.tok0 * H * a->dv * es;
  s.g = w + L.g + p.tok0 * H * (a->gate_per_head ? 1 : a->dk) * es;
  s.gate_per_head = a->gate_per_head;
  s.b = w + L.b + p.tok0 * H * es;
  s.scale = a->scale;
  s.o = w + L.o + p.tok0 * H * a->dv * es;
  s.scan_segments = 1;  // the pieces already cut the chain; keep kda_prefill's plain path
  float* init = a->initial_state ? reinterpret_cast<float*>(w + L.init) : nullptr;
  float* fin = reinterpret_cast<float*>(w + L.fin);
  float* carry = reinterpret_cast<float*>(w + L.carry);
  if (p.split) {
    // one sequence: piece i starts where piece i-1 ended
    s.initial_state = i == 0 ? init : carry + ((i - 1) & 1) * state;
    s.final_state = i + 1 == pieces.size() ? fin : carry + (i & 1) * state;
  } else {
    s.initial_state = init ? init + p.seq0 * state : nullptr;
    s.final_state = fin + p.seq0 * state;
  }
  return s;
}

// Offsets of the device copies inside the workspace; the prefill workspace
// comes first, so that its status word (offset 0) is the workspace's.
HostLayout host_layout(const kda_prefill_host_args* a, const std::vector<Piece>& pieces) {
  const int64_t T = a->total_tokens, H = a->num_heads, N = a->num_seqs;
  const int64_t es = a->in_dtype == KDA_BF16 ? 2 : 4;
  const size_t state = (size_t)H * a->dk * a->dv * sizeof(float);
  HostLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.q = take((size_t)T * H * a->dk * es);
  L.k = take((size_t)T * H * a->dk * es);
  L.v = take((size_t)T * H * a->dv * es);
  L.g = take((size_t)T * H * (a->gate_per_head ? 1 : a->dk) * es);
  L.b = take((size_t)T * H * es);
  L.o = take((size_t)T * H * a->dv * es);
  L.init = take(a->initial_state ? N * state : 0);
  L.fin = take(N * state);
  L.carry = take(2 * state);
  L.cu_all = take((size_t)(N + 1) * sizeof(int64_t));
  L.cu_piece = take((size_t)(N + pieces.size()) * sizeof(int64_t));
  L.acc = take(sizeof(int32_t));
  // the largest prefill workspace of any piece, its tensors placed as they
  // will be relative to a 256-byte aligned base (alignment picks the path)
  char* const stand_in = reinterpret_cast<char*>((uintptr_t)1 << 20);
  size_t pws = 0;
  for (size_t i = 0; i < pieces.size(); ++i) {
    const kda_prefill_args s = piece_args(a, L, stand_in, pieces, i);
    const size_t need = kda_prefill_workspace_size(&s);
    if (need == 0) return HostLayout{};
    pws = need > pws ? need : pws;
  }
  L.pws = 0;
  L.pws_bytes = align_up(pws, 256);
  for (size_t* f : {&L.q, &L.k, &L.v, &L.g, &L.b, &L.o, &L.init, &L.fin, &L.carry, &L.cu_all,
                    &L.cu_piece, &L.acc})
    *f += L.pws_bytes;
  L.total = L.pws_bytes + off;
  return L;
}

// cu_seqlens of piece i on the device: {0, len} for a cut of one sequence,
// else the piece's sequences rebased to its first token.
__global__ void piece_cu(const int64_t* __restrict__ cu_all, int64_t* __restrict__ dst, int32_t seq0,
                         int32_t nseq, int64_t len, int32_t split) {
  for (int i = threadIdx.x; i <= nseq; i += blockDim.x)
    dst[i] = split ? (i == 0 ? 0 : len) : cu_all[seq0 + i] - cu_all[seq0];
}
// After each piece: acc |= status; status = acc (the next piece's planning
// kernel clears status, so it ends as the OR over all pieces).
__global__ void piece_status(int32_t* __restrict__ status, int32_t* __restrict__ acc, int32_t first) {
  if (threadIdx.x == 0) {
    const int32_t v = (first ? 0 : *acc) | *status;
    *acc = v;
    *status = v;
  }
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_prefill_host_workspace_size(const kda_prefill_host_args* a) {
  if (validate_host(a) != KDA_OK) return 0;
  const std::vector<Piece> pieces = plan_pieces(a);
  return host_layout(a, pieces).total;
}

extern "C" kda_status_t kda_prefill_host(const kda_prefill_host_args* a, void* ws, size_t ws_bytes,
                                         void* stream_) {
  kda_status_t st = validate_host(a);
  if (st != KDA_OK) return st;
  if (!a->copy_in_stream || !a->copy_out_stream || a->copy_in_stream == stream_ ||
      a->copy_out_stream == stream_ || a->copy_in_stream == a->copy_out_stream)
    return KDA_ERR_INVALID_ARG;
  const std::vector<Piece> pieces = plan_pieces(a);
  char* w = static_cast<char*>(ws);
  const HostLayout L = host_layout(a, pieces);
  if (L.total == 0) return KDA_ERR_INVALID_ARG;
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255) != 0)
    return KDA_ERR_WORKSPACE;

  cudaStream_t cs = static_cast<cudaStream_t>(stream_);
  cudaStream_t in = static_cast<cudaStream_t>(a->copy_in_stream);
  cudaStream_t out = static_cast<cudaStream_t>(a->copy_out_stream);
  const size_t np = pieces.size();
  const int64_t H = a->num_heads, N = a->num_seqs, es = a->in_dtype == KDA_BF16 ? 2 : 4;
  const size_t state = (size_t)H * a->dk * a->dv * sizeof(float);

  // events: start, per piece (inputs in, computed), all out
  std::vector<cudaEvent_t> ev(2 * np + 2, nullptr);
  cudaError_t e = cudaSuccess;
  for (auto& x : ev)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
  cudaEvent_t ev_start = ev[0], ev_out = ev[1];
  cudaEvent_t* ev_in = ev.data() + 2;
  cudaEvent_t* ev_done = ev.data() + 2 + np;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  auto h2d = [&](size_t dst, const void* src, size_t bytes) {
    if (bytes) ok(cudaMemcpyAsync(w + dst, src, bytes, cudaMemcpyHostToDevice, in));
  };

  // the copy streams start after the work already queued on `stream` (which
  // may still be reading this workspace)
  if (e == cudaSuccess) {
    ok(cudaEventRecord(ev_start, cs));
    ok(cudaStreamWaitEvent(in, ev_start, 0));
    ok(cudaStreamWaitEvent(out, ev_start, 0));
  }
  h2d(L.cu_all, a->cu_seqlens, (size_t)(N + 1) * sizeof(int64_t));
  if (a->initial_state) h2d(L.init, a->initial_state, N * state);
  const char* hq = static_cast<const char*>(a->q);
  const char* hk = static_cast<const char*>(a->k);
  const char* hv = static_cast<const char*>(a->v);
  const char* hg = static_cast<const char*>(a->g);
  const char* hb = static_cast<const char*>(a->b);
  // b (2 bytes a token-head) in one copy: each copy costs the engine a
  // couple of microseconds, so the pieces carry only q, k, g, v
  h2d(L.b, hb, (size_t)a->total_tokens * H * es);
  for (size_t i = 0; i < np && e == cudaSuccess; ++i) {
    const int64_t t0 = pieces[i].tok0, n = pieces[i].tok1 - pieces[i].tok0;
    const size_t rk = (size_t)H * a->dk * es, rv = (size_t)H * a->dv * es;
    const size_t rg = a->gate_per_head ? (size_t)H * es : rk;
    h2d(L.q + t0 * rk, hq + t0 * rk, n * rk);
    h2d(L.k + t0 * rk, hk + t0 * rk, n * rk);
    h2d(L.g + t0 * rg, hg + t0 * rg, n * rg);
    h2d(L.v + t0 * rv, hv + t0 * rv, n * rv);
    ok(cudaEventRecord(ev_in[i], in));
  }
  char* ho = static_cast<char*>(a->o);
  int32_t* status = reinterpret_cast<int32_t*>(w + L.pws);  // kda_prefill's status word
  for (size_t i = 0; i < np && e == cudaSuccess; ++i) {
    const Piece& p = pieces[i];
    ok(cudaStreamWaitEvent(cs, ev_in[i], 0));
    piece_cu<<<1, 128, 0, cs>>>(reinterpret_cast<const int64_t*>(w + L.cu_all),
                                reinterpret_cast<int64_t*>(w + L.cu_piece) + p.cu_off, p.seq0,
                                p.nseq, p.tok1 - p.tok0, p.split ? 1 : 0);
    if (!ok(cudaGetLastError())) break;
    const kda_prefill_args s = piece_args(a, L, w, pieces, i);
    st = kda_prefill(&s, w + L.pws, L.pws_bytes, cs);
    if (st != KDA_OK) break;
    piece_status<<<1, 32, 0, cs>>>(status, reinterpret_cast<int32_t*>(w + L.acc), i == 0);
    ok(cudaGetLastError());
    ok(cudaEventRecord(ev_done[i], cs));
    ok(cudaStreamWaitEvent(out, ev_done[i], 0));
    const size_t ro = (size_t)H * a->dv * es;
    if (p.tok1 > p.tok0)
      ok(cudaMemcpyAsync(ho + p.tok0 * ro, w + L.o + p.tok0 * ro, (p.tok1 - p.tok0) * ro,
                         cudaMemcpyDeviceToHost, out));
  }
  if (a->final_state && e == cudaSuccess && st == KDA_OK)
    ok(cudaMemcpyAsync(a->final_state, w + L.fin, N * state, cudaMemcpyDeviceToHost, out));
  // `stream` continues only after everything, copies out included
  if (ev_out) {
    if (cudaEventRecord(ev_out, out) == cudaSuccess) cudaStreamWaitEvent(cs, ev_out, 0);
  }
  for (auto& x : ev)
    if (x) cudaEventDestroy(x);  // released once the work that records it has run
  if (st != KDA_OK) return st;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
