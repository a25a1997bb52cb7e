// kda_plan.cu -- builds the chunk table of a prefill call on the device.
//
// The chunked prefill ("Kimi K3: The Manos, The Mythos, The Legendos":
// FlashKDA unrolls the recurrence in chunks) needs the sequence cut into
// runs of at most KDA_CHUNK tokens.  Cut points of sequence s are the
// multiples of KDA_CHUNK, every boundary position (snapshots must fall on a
// chunk end, as the snapshot of a prompt boundary is the state after its last
// token, same page, Context) and the sequence end.  Snapshot interval
// multiples are multiples of KDA_CHUNK and need no extra cut.
//
// Two launches, no host synchronisation:
//   plan_sequences (one CTA): validates cu_seqlens and boundaries, counts the
//     aligned segments and chunks per sequence, prefix-sums them.
//   plan_fill (grid over aligned segments): writes the chunk entries.
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int64_t lower_bound_i64(const int64_t* a, int64_t lo, int64_t hi,
                                                   int64_t x) {
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ int64_t upper_bound_i64(const int64_t* a, int64_t lo, int64_t hi,
                                                   int64_t x) {
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Block-wide exclusive scan of one value per thread; `total` receives the
// sum.  A shuffle scan inside each warp, the warps' sums scanned by warp 0
// through shared memory (sh: one entry per warp), two barriers.
__device__ int64_t block_exclusive_scan(int64_t x, int64_t* sh, int64_t& total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) sh[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int64_t w = sh[lane];  // kPlanThreads / 32 == 32 warps
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    sh[lane] = w;  // inclusive sums of the warps
  }
  __syncthreads();
  const int64_t before = warp > 0 ? sh[warp - 1] : 0;
  total = sh[kPlanThreads / 32 - 1];
  __syncthreads();  // every thread has read before sh is reused
  return before + incl - x;
}
static_assert(kPlanThreads == 32 * 32, "the scan has one warp sum per lane of warp 0");

// Per-sequence validation, counts and prefix sums (whole block).
__device__ void plan_sequences(const PlanParams& p, int64_t* sh, int32_t& flags) {
  const int tid = threadIdx.x;
  int64_t seg_carry = 0, chunk_carry = 0;
  for (int32_t base = 0; base < p.num_seqs; base += kPlanThreads) {
    const int32_t s = base + tid;
    int64_t nseg = 0, nchunk = 0;
    if (s < p.num_seqs) {
      int64_t c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
      int64_t len = c1 - c0;
      bool ok = (c0 >= 0) && (len >= 0) && (c1 <= p.total_tokens) && (s > 0 || c0 == 0);
      if (!ok) { flags |= kFlagBadSeqlens; len = 0; }
      int64_t b0 = 0, b1 = 0;
      if (p.boundary_pos) {
        b0 = p.cu_boundaries[s];
        b1 = p.cu_boundaries[s + 1];
        bool bok = b0 >= 0 && b1 >= b0 && b1 <= p.num_boundaries;
        for (int64_t i = b0; bok && i < b1; ++i) {
          int64_t x = p.boundary_pos[i];
          if (x < 1 || x > len || (i > b0 && x <= p.boundary_pos[i - 1])) bok = false;
        }
        if (!bok) { flags |= kFlagBadBoundaries; b0 = b1 = 0; }
      }
      // empty range (b0 == b1): the prefix arrays are neither written nor read
      p.seq_bnd[2 * s] = b0;
      p.seq_bnd[2 * s + 1] = b1;
      // prefix counts of non-aligned boundaries (they add a cut) and of
      // boundaries that are not interval multiples (they add a snapshot);
      // entry i + s for i in [b0, b1] (the +s keeps sequences apart)
      int32_t na = 0, nm = 0;
      int64_t extra = 0;
      if (b1 > b0) {
        for (int64_t i = b0; i < b1; ++i) {
          p.bnd_nonaligned[i + s] = na;
          p.bnd_nonmult[i + s] = nm;
          const int64_t x = p.boundary_pos[i];
          if (x % kChunk != 0) { ++na; if (x < len) ++extra; }
          if (p.snapshot_interval <= 0 || x % p.snapshot_interval != 0) ++nm;
        }
        p.bnd_nonaligned[b1 + s] = na;
        p.bnd_nonmult[b1 + s] = nm;
      }
      nseg = (len + kChunk - 1) / kChunk;
      nchunk = nseg + extra;
      p.seq_len[s] = len;
    }
    int64_t seg_total = 0, ch_total = 0;
    const int64_t seg_ex = block_exclusive_scan(nseg, sh, seg_total);
    const int64_t ch_ex = block_exclusive_scan(nchunk, sh, ch_total);
    if (s < p.num_seqs) {
      p.seq_seg_begin[s] = seg_carry + seg_ex;
      p.seq_chunk_begin[s] = chunk_carry + ch_ex;
    }
    seg_carry += seg_total;
    chunk_carry += ch_total;
  }
  if (tid == 0) {
    int64_t total = chunk_carry;
    if (total > p.max_chunks) { flags |= kFlagChunkOverflow; total = 0; }
    p.seq_seg_begin[p.num_seqs] = seg_carry;
    p.seq_chunk_begin[p.num_seqs] = chunk_carry;
    p.meta->total_chunks = total;
  }
}

// Writes the chunk entries of aligned 64-token segment gidx; bad |= 1 on a
// snapshot slot outside the caller's snapshot buffer.
__device__ void fill_segment(const PlanParams& p, int64_t gidx, int32_t& bad) {
  // sequence owning this aligned segment: largest s with seg_begin[s] <= gidx
  int32_t lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) >> 1;
    if (p.seq_seg_begin[mid] <= gidx) lo = mid; else hi = mid - 1;
  }
  const int32_t s = lo;
  const int64_t m = gidx - p.seq_seg_begin[s];
  const int64_t len = p.seq_len[s];
  const int64_t tok_base = p.cu_seqlens[s];
  const int64_t b0 = p.seq_bnd[2 * s], b1 = p.seq_bnd[2 * s + 1];
  const bool has_b = p.boundary_pos != nullptr && b1 > b0;
  const int64_t seg0 = m * kChunk;
  const int64_t seg1 = seg0 + kChunk < len ? seg0 + kChunk : len;
  int64_t j = has_b ? lower_bound_i64(p.boundary_pos, b0, b1, seg0 + 1) : 0;
  int64_t ci = p.seq_chunk_begin[s] + m + (has_b ? p.bnd_nonaligned[j + s] : 0);
  const int64_t snap_lo = p.cu_snapshots ? p.cu_snapshots[s] : 0;
  const int64_t snap_hi = p.cu_snapshots ? p.cu_snapshots[s + 1] : 0;
  int64_t start = seg0;
  while (start < seg1) {
    int64_t end = seg1;
    if (has_b && j < b1 && p.boundary_pos[j] < seg1) end = p.boundary_pos[j];
    // snapshot slot of the state after `end` tokens
    int32_t slot = -1;
    if (p.cu_snapshots) {
      bool is_mult = p.snapshot_interval > 0 && end % p.snapshot_interval == 0;
      int64_t jb = has_b ? upper_bound_i64(p.boundary_pos, b0, b1, end) : 0;
      bool is_bnd = has_b && jb > b0 && p.boundary_pos[jb - 1] == end;
      if (is_mult || is_bnd) {
        int64_t rank = (p.snapshot_interval > 0 ? end / p.snapshot_interval : 0) +
                       (has_b ? p.bnd_nonmult[jb + s] : 0) - 1;
        const int64_t sl = snap_lo + rank;
        if (sl < snap_lo || sl >= snap_hi) {
          bad = 1;
        } else if (p.slot_map) {
          // snapshot sl goes to the row the map gives (negative: not written)
          const int32_t row = sl < p.map_len ? p.slot_map[sl] : INT32_MAX;
          if (row < 0) slot = -1;
          else if (row < p.num_snapshots) slot = row;
          else bad = 1;
        } else if (sl < p.num_snapshots) {
          slot = (int32_t)sl;
        } else {
          bad = 1;
        }
      }
    }
    if (ci < p.max_chunks) {
      Chunk c;
      c.tok0 = tok_base + start;
      c.seq = s;
      c.len = (int32_t)(end - start);
      c.snap_slot = slot;
      c.flags = (start == 0 ? kChunkFirst : 0) | (end == len ? kChunkLast : 0);
      c.pos = start;
      p.chunks[ci] = c;
    }
    ++ci;
    if (has_b && j < b1 && p.boundary_pos[j] == end) ++j;
    start = end;
  }
}

// One CTA: clears the status word (and the words of zero_words), plans the
// sequences, writes every chunk entry, and marks the unused tail of the table
// (len = 0) so that the per-chunk kernels can read their entry without
// consulting the totals.  The intra-chunk kernel after it may be launched as
// its programmatic dependent: it is let start at once, and it waits for this
// kernel's results before it reads them.
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(PlanParams p) {
  __shared__ int64_t sh[kPlanThreads];
  __shared__ int32_t cnt[kPlanThreads];  // chunk counts of the sequences (their order)
  __shared__ int32_t shf;
  const int tid = threadIdx.x;
  pdl_launch_dependents();
  if (tid == 0) {
    *p.status = 0;
    shf = 0;
  }
  // (a multiple of 4 words, 16-byte aligned)
  for (int64_t i = tid; i < p.n_zero_words / 4; i += kPlanThreads)
    reinterpret_cast<uint4*>(p.zero_words)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  int32_t flags = 0;
  plan_sequences(p, sh, flags);
  __syncthreads();  // totals written by thread 0 are visible to the block
  const int64_t total = p.meta->total_chunks;
  const int64_t total_segs = total > 0 ? p.seq_seg_begin[p.num_seqs] : 0;
  int32_t bad = 0;
  for (int64_t gidx = tid; gidx < total_segs; gidx += kPlanThreads) fill_segment(p, gidx, bad);
  if (bad) flags |= kFlagBadBoundaries;
  Chunk empty{};
  empty.snap_slot = -1;
  for (int64_t ci = total + tid; ci < p.max_chunks; ci += kPlanThreads) p.chunks[ci] = empty;
  if (flags) atomicOr(&shf, flags);
  // the sequences by chunk count, longest first: thread s finds the rank of
  // sequence s among the counts in shared memory (up to kPlanThreads
  // sequences; more keep their own order)
  if (p.seq_order) {
    const int32_t N = p.num_seqs;
    if (N <= kPlanThreads) {
      int32_t mine = 0;
      if (tid < N) {
        const int64_t n = p.seq_chunk_begin[tid + 1] - p.seq_chunk_begin[tid];
        mine = n < INT32_MAX ? (int32_t)n : INT32_MAX;
        cnt[tid] = mine;
      }
      __syncthreads();
      if (tid < N) {
        int32_t rank = 0;
        for (int32_t t = 0; t < N; ++t) {
          const int32_t o = cnt[t];
          rank += (o > mine || (o == mine && t < tid)) ? 1 : 0;
        }
        p.seq_order[rank] = tid;
      }
    } else {
      for (int32_t s = tid; s < N; s += kPlanThreads) p.seq_order[s] = s;
    }
  }
  __syncthreads();
  if (tid == 0 && shf) atomicOr(p.status, shf);
}

}  // namespace

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
