/*
 * kda.h -- C ABI of libkda, a GB300 (sm_103a) library for the Kimi Delta
 * Attention (KDA) recurrence.
 *
 * The operation.  Each attention head keeps one fixed-size fp32 state
 * S in R^{dk x dv}.  For every token t of a sequence:
 *
 *     q^ = q_t / max(|q_t|, 1e-6)           k^ = k_t / max(|k_t|, 1e-6)
 *     alpha_t = exp(-softplus(g_t))  (per key channel, dk values)
 *     beta_t  = sigmoid(b_t)         (one value per token and head)
 *     S_t = (I - beta_t k^ k^T) Diag(alpha_t) S_{t-1} + beta_t k^ v_t^T
 *     o_t = scale * S_t^T q^
 *
 *   - "From KV Cache to Depth Attention: The Bottlenecks Kimi K3 Had to
 *     Break", Technical Details: the state predicts the value from its
 *     memory and writes back only the difference; alpha is retention, beta
 *     update strength, and each feature channel has its own timescale.
 *   - "Kimi K3: The Manos, The Mythos, The Legendos", bullet list: delta
 *     rule plus a forget gate made diagonal; L2-normalised queries and keys;
 *     FlashKDA's chunked unrolling gives linear prefill and constant-cost
 *     decode.  Its Context section: the serving engine keeps state snapshots
 *     at prompt boundaries so that later requests can resume from them.
 *
 * Conventions shared by every call.
 *   - Every tensor is caller-owned device memory, row-major and contiguous,
 *     token-major: q, k, g [T, H, dk] (g [T, H] with gate_per_head);
 *     v, o [T, H, dv]; b [T, H]; states
 *     [.., H, dk, dv] fp32.  No call allocates device memory.  The library
 *     keeps no mutable global state, with one exception: the fixed workspace
 *     array behind kda_prefill_noalloc (see there).  The prefix cache's host
 *     index lives in the object the caller creates.  Calls from several host
 *     threads are safe (kda_prefill_noalloc calls share its array: see there).
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream).  Arguments are validated on the host before any
 *     launch; on an error nothing is launched and the status says why.
 *   - Values that live on the device (cu_seqlens, boundary positions, slot
 *     indices) are checked by the kernels: a malformed value raises a flag
 *     in the workspace status word (see kda_prefill_device_status) and the
 *     affected sequence is skipped; no kernel traps.
 *   - Outputs must not alias inputs; snapshots, initial and final states must
 *     not overlap one another.
 *   - No C++ exception crosses this boundary.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent argument  */
  KDA_ERR_UNSUPPORTED = 2, /* head size or dtype this build does not cover   */
  KDA_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned     */
  KDA_ERR_CUDA = 4,        /* a CUDA launch or query failed                  */
  KDA_ERR_TIMEOUT = 5,     /* a bounded device-side wait expired             */
  KDA_ERR_DEVICE_DATA = 6  /* a device-side index array was malformed        */
} kda_status_t;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype_t;

/* Chunk length of the chunked prefill (tokens). */
#define KDA_CHUNK 64

/*
 * The layer steps on either side of the recurrence (optional).
 *
 * "Kimi K3: The Manos, The Mythos, The Legendos" (bullet on the stability
 * details) names a short convolution on q, k and v and a per-head output
 * forget gate around the recurrence.  The pages give neither formula; the
 * readings implemented here:
 *
 *   Short convolution, per channel c of each of q, k, v (x one of them):
 *     y_t[c] = sum_{j < conv_width} w[j][h][c] * x_{t-j}[c]
 *   a causal depthwise convolution along the tokens of one sequence; tap j
 *   multiplies the input j tokens back.  Inputs before the first token of a
 *   sequence come from its window (the conv_width - 1 inputs that preceded
 *   it), zeros when no window is given.  With conv_silu, y <- y * sigmoid(y).
 *   The result is rounded to in_dtype (the precision a separate layer would
 *   store it in) and is what the recurrence then takes as q, k, v (so the
 *   L2 normalisation of q and k follows the convolution).
 *
 *   Output gate: o_t <- o_t * sigmoid(r_t), with r [T, H, dv] (a gate per
 *   value channel) or [T, H] (out_gate_per_head: one gate per token and
 *   head), applied after scale and before the rounding of o.
 *
 * Windows.  A window holds the raw (unconvolved) inputs of the last
 * conv_width - 1 tokens, oldest first: [rows, conv_width - 1, H, d] in
 * in_dtype, row = sequence (prefill) or state slot (decode).  conv_in gives
 * the windows before the call, conv_out receives those after it (a sequence
 * shorter than the window keeps the older entries of its input window).  In
 * the prefill, conv_out may be the same buffer as conv_in (updated in place)
 * but must not partly overlap it; in the decode both are indexed by the
 * row's state slot and may be the same buffer.  Snapshots hold only S: a
 * prefill that resumes at a snapshot position p passes the raw inputs of
 * tokens p - conv_width + 1 .. p - 1 as its window.
 */
#define KDA_CONV_MAX 4

typedef struct {
  int32_t conv_width;          /* 0 = no convolution, else 1..KDA_CONV_MAX taps  */
  int32_t conv_silu;           /* nonzero: SiLU after the convolution            */
  const float* conv_w[3];      /* taps of q, k, v: device [conv_width, H, d] fp32
                                  (d = dk, dk, dv); all three when conv_width > 0 */
  const void* conv_in[3];      /* windows of q, k, v before the call, or NULL
                                  (zeros); each may be NULL on its own           */
  void* conv_out[3];           /* windows of q, k, v after the call, or NULL     */
  const void* out_gate;        /* device gate logits, in_dtype: [T, H, dv], or
                                  [T, H] with out_gate_per_head; NULL = no gate   */
  int32_t out_gate_per_head;
} kda_layer_args;

/*
 * Prefill over packed variable-length sequences.
 *
 * Sequence s holds packed tokens [cu_seqlens[s], cu_seqlens[s+1]).  Each
 * (sequence, head) starts from initial_state (or zeros), runs the
 * recurrence over its tokens, writes o for every token, its final state and
 * the snapshots it owns.
 *
 * Snapshot positions (seq-relative token counts p, the state after p tokens,
 * as in "Kimi K3: The Manos, The Mythos, The Legendos", Context) of sequence
 * s are the sorted, de-duplicated union of
 *   { p : p % snapshot_interval == 0, 0 < p <= len }   (if interval > 0)
 *   boundary_pos[cu_boundaries[s] .. cu_boundaries[s+1])  (if given)
 * Snapshot j of sequence s goes to snapshots[cu_snapshots[s] + j].
 * kda_snapshot_plan() computes cu_snapshots on the host.
 */
typedef struct {
  int32_t num_seqs;            /* N >= 1                                          */
  int32_t num_heads;           /* H >= 1                                          */
  int32_t dk, dv;              /* each in {16, 32, 64, 128, 256}                  */
  int64_t total_tokens;        /* T = cu_seqlens[N]; host-known upper bound, >= 0 */
  const int64_t* cu_seqlens;   /* device [N+1], cu[0] = 0, non-decreasing         */
  kda_dtype_t in_dtype;        /* dtype of q, k, v, g, b and of o                 */
  const void* q;               /* device [T, H, dk]                               */
  const void* k;               /* device [T, H, dk]                               */
  const void* v;               /* device [T, H, dv]                               */
  const void* g;               /* device [T, H, dk], decay logit                  */
  const void* b;               /* device [T, H], update logit                     */
  float scale;                 /* o = scale * S^T q^; 1.0 is the plain recurrence */
  const float* initial_state;  /* device [N, H, dk, dv] or NULL (zeros)           */
  void* o;                     /* device [T, H, dv], in_dtype                     */
  float* final_state;          /* device [N, H, dk, dv] or NULL                   */
  int64_t snapshot_interval;   /* 0 = off, else a positive multiple of KDA_CHUNK  */
  const int64_t* boundary_pos; /* device, per sequence strictly increasing in [1, len], or NULL */
  const int64_t* cu_boundaries;/* device [N+1] offsets into boundary_pos (NULL iff boundary_pos is) */
  int64_t num_boundaries;      /* host-known total entries of boundary_pos (0 if NULL) */
  const int64_t* cu_snapshots; /* device [N+1] snapshot slot offsets, or NULL if no snapshots */
  float* snapshots;            /* device [num_snapshots, H, dk, dv] or NULL       */
  int64_t num_snapshots;       /* host-known rows of `snapshots`; a slot at or past
                                  it is not written and raises status flag 2     */
  void* const* phase_events;   /* NULL, or KDA_PREFILL_PHASES + 1 cudaEvent_t the call
                                  records on `stream` before the first phase and after
                                  each phase (chunk planning, intra-chunk,
                                  inter-chunk), for per-kernel timing             */
  int32_t scan_segments;       /* segment scan: 0 = automatic, 1 = off, P >= 2 = P
                                  segments (see below); at most 64                */
  const int32_t* snapshot_slot_map; /* device [snapshot_map_len] or NULL: snapshot j of
                                  the call (j counted through cu_snapshots) goes to row
                                  snapshot_slot_map[j] of `snapshots` instead of row
                                  j; a negative entry skips it; a row at or past
                                  num_snapshots, or j at or past snapshot_map_len,
                                  raises status flag 2 (for a prefix cache choosing
                                  pool rows, see kda_prefix_cache_reserve)        */
  int64_t snapshot_map_len;    /* entries of snapshot_slot_map (0 if NULL)       */
  int64_t wait_limit_ns;       /* 0 = 1 s: how long a kernel's bounded wait on a
                                  copy or an MMA lasts before the kernel gives up,
                                  raises status flag 8 and winds down (its copies
                                  and MMAs in flight are still awaited, with the
                                  1 s limit).  A short limit exercises that path. */
  int32_t gate_per_head;       /* 0: g is [T, H, dk], a decay per key channel (KDA);
                                  1: g is [T, H], one decay per token and head (the
                                  gated delta rule: "Kimi K3: The Manos, The
                                  Mythos, The Legendos" bullet on KDA as online
                                  learning -- a forget gate, which KDA makes
                                  diagonal); the result is that of a per-channel g
                                  holding the same value in every channel       */
  const kda_layer_args* layer; /* host pointer, or NULL: the short convolution and
                                  output gate (above); read during the call only.
                                  Windows are [N, conv_width - 1, H, d]          */
  int32_t schedule;            /* KDA_SCHEDULE_SEPARATE (1): the intra-chunk and
                                  inter-chunk kernels one after the other;
                                  KDA_SCHEDULE_FUSED (2): the fused kernel where it
                                  applies (see below), else the two kernels;
                                  KDA_SCHEDULE_OVERLAP (3): the overlapped kernels
                                  where they apply (see below), else the two
                                  kernels; KDA_SCHEDULE_AUTO (0): the overlapped
                                  kernels where they apply, else the two kernels.
                                  All give the same results, bit for bit        */
} kda_prefill_args;

#define KDA_SCHEDULE_AUTO 0
#define KDA_SCHEDULE_SEPARATE 1
#define KDA_SCHEDULE_FUSED 2
#define KDA_SCHEDULE_OVERLAP 3

/*
 * Segment scan.  The inter-chunk recurrence of one sequence is a chain over
 * its chunks, and each (sequence, head) runs it on a few SMs only.  When the
 * call has few heads and one long sequence, the chain is cut into P
 * chunk-aligned segments.  Every segment runs in parallel twice from a
 * known start: from the zero state, giving its state offset B_s, and from
 * the identity with v = 0, giving its transition map A_s (dk x dk), so that
 * S_end(s) = A_s S_start(s) + B_s, the recurrence being affine in S.  A
 * short serial combine forms the true start states, and a second parallel
 * pass over the segments writes o and the final state.  The chunk algebra
 * itself runs once.  This is a reading of the recurrence's linearity, not a
 * step the pages give.  It applies on the tensor-core path, to one sequence
 * without snapshots or boundary positions; otherwise scan_segments is
 * ignored.  Automatic (0) uses it when 8 * num_heads * P CTAs fit the GPU
 * with P >= 3 segments of >= 16 chunks each.  The results match the unsplit
 * chain to rounding (fp32 state combine), not bit for bit.
 */

/*
 * Fused prefill (schedule = KDA_SCHEDULE_FUSED).  On the tensor-core path the
 * intra-chunk step (K2) and the inter-chunk chains (K3) run as one kernel of
 * two CTAs per SM: a CTA either runs the chain of one (sequence, head,
 * 32-column slice of the state) or a pipeline of (chunk, head) items taken in
 * chunk order.  Each record is published once written; a chain copies it as
 * soon as it sees it, so the chains run while the items are made (and read
 * the records from L2 while they keep up).  Pipelines never wait
 * for chains and the chains are placed after the pipelines they read, so no
 * wait depends on the CTAs being resident together.  It applies without the
 * segment scan when the chains (num_seqs x num_heads x dv / 32) are at most
 * as many as the SMs.  A chain waits for a record at most the longer of
 * wait_limit_ns and 1 s.  Measured on GB300 it is slower than the two kernels
 * (a chain step takes about twice as long on an SM shared with another CTA
 * as on an SM of its own), so the automatic choice does not take it.  With
 * phase_events, the intra-chunk phase holds the fused kernel and the
 * inter-chunk phase only what follows it.
 */

/*
 * Overlapped prefill (schedule = KDA_SCHEDULE_OVERLAP or AUTO).  On the
 * tensor-core path the intra-chunk kernel (K2) takes its (chunk, head) items
 * in chunk order from a counter on every SM until most are taken; then its
 * CTAs leave every SM but a few, which make the remaining records.  The
 * inter-chunk kernel (K3) is launched as K2's programmatic dependent: its
 * chains (one per head and 32-column slice of the state, each on an SM of
 * its own) start on the SMs K2 leaves, and read each record once K2 has
 * published it, while the last ones are still being made.  A chain needs
 * the record of chunk j only j chain steps after it starts, so the chains
 * no longer wait for the last item.  It applies on the tensor-core path
 * without the segment scan, to one sequence whose chains
 * (num_heads x dv / 32) leave at least 8 SMs for K2, with a wait limit of
 * 0 or at least 100 us.  A chain waits for a record at most the longer of
 * wait_limit_ns and 1 s.  With phase_events, the intra-chunk phase holds
 * both kernels.
 */

/* The path kda_prefill takes for these arguments on a GPU with sm_count SMs
 * (0: the current device, which must then be present).  Host-side fields
 * only; -1 for invalid arguments or a failed device query. */
#define KDA_PATH_CUDA_CORES 0    /* fp32 CUDA-core kernels                  */
#define KDA_PATH_SEPARATE 1      /* tensor cores, K2 then K3                 */
#define KDA_PATH_FUSED 2         /* tensor cores, the fused kernel           */
#define KDA_PATH_SEGMENT_SCAN 3  /* tensor cores, the segment scan           */
#define KDA_PATH_OVERLAP 4       /* tensor cores, K2 and K3 overlapped       */
int32_t kda_prefill_schedule(const kda_prefill_args* args, int32_t sm_count);

/* Number of timed phases of kda_prefill (see phase_events). */
#define KDA_PREFILL_PHASES 3

/* Bytes of device workspace kda_prefill needs for these arguments (reads
 * only host-side fields).  Returns 0 if the arguments are invalid. */
size_t kda_prefill_workspace_size(const kda_prefill_args* args);

/* Runs the prefill.  ws: device buffer of at least
 * kda_prefill_workspace_size(args) bytes, 256-byte aligned, owned by the
 * caller and not used by another call in flight.  The path is chosen by the
 * arguments: bf16 inputs with dk <= 128 and dv in {32, 64, 128} run on the
 * tcgen05 tensor-core kernels (a head narrower than 128 channels runs
 * zero-padded to 128, at the cost of a 128-channel head; with the short
 * convolution only dk = dv = 128); every other supported shape runs on fp32
 * CUDA-core kernels (heads of 256 channels on a variant that takes 128
 * channels at a time). */
kda_status_t kda_prefill(const kda_prefill_args* args, void* ws, size_t ws_bytes,
                         void* stream);

/* kda_prefill for callers that cannot allocate device memory at the point of
 * the call (all of HBM reserved up front for state pools, a host framework
 * that owns every allocation, or a path where an allocation would
 * synchronise the device).  This entry has no counterpart on the pages; it
 * is a deployment convenience.  It runs the same kernels as kda_prefill on a
 * workspace held in a fixed 64 MiB (67108864-byte) __device__ array inside
 * this library, which every GPU that loads the library keeps until the
 * process exits; the call itself allocates nothing.
 *   - Arguments whose kda_prefill_workspace_size exceeds 64 MiB are rejected
 *     with KDA_ERR_WORKSPACE before any launch (for example about 650
 *     (chunk, head) pairs on the bf16 dk = dv = 128 path).
 *   - A call made outside stream capture looks up the array's device
 *     address on the current device (cudaGetSymbolAddress) and remembers it
 *     for that device; a call made while `stream` is capturing uses the
 *     remembered address.  Make the first call on each device before any
 *     stream capture (a capturing call with none remembered returns
 *     KDA_ERR_CUDA).
 *   - All calls share the array: calls whose kernels overlap on the GPU race
 *     on it, so serialise them (one stream, or events).  Nothing in it needs
 *     to start at zero.  kda_prefill_noalloc_device_status reads its status
 *     word (the device-side flags of the last call). */
kda_status_t kda_prefill_noalloc(const kda_prefill_args* args, void* stream);

/* The device status word of the last kda_prefill_noalloc on the current
 * device (the same flags as kda_prefill_device_status), copied to *out
 * (host), synchronising `stream`.  Allocates nothing.  No counterpart on the
 * pages: it completes kda_prefill_noalloc, whose workspace the caller cannot
 * name. */
kda_status_t kda_prefill_noalloc_device_status(int32_t* out, void* stream);

/*
 * kda_prefill from HOST buffers, end to end: the inputs are copied to the
 * device, the prefill runs, and o and the final state are copied back, with
 * the copies of one piece of the batch overlapping the prefill of another.
 * The operation and its results are those of kda_prefill without the
 * segment scan (the same kernels, bit for bit); only where the tensors live
 * differs.  This entry has no
 * counterpart on the pages; it is the call a serving host makes when a
 * prompt's q, k, v, g, b sit in host memory.
 *
 * Pipelining.  The batch is cut into about `segments` equal pieces (0 = one
 * per 48 chunks of the batch, at most 4; 1 = no cut).  A single sequence is
 * cut at chunk boundaries, and the end of it into a few halving pieces (1/8,
 * 1/4, 1/2 of a piece) so that the prefill and copy-out of the last piece,
 * which nothing overlaps, are short.  Piece p starts from the fp32 final
 * state of piece p-1: the same arithmetic as one call, because the chunked
 * recurrence restarts its chunk algebra at every chunk boundary anyway.  A
 * batch of several sequences is cut only between sequences.  Piece p+1 is copied in on
 * copy_in_stream while piece p is computed on `stream`; piece p's o is copied
 * out on copy_out_stream as soon as it is ready.
 *
 * Memory.  All host buffers are caller-owned, row-major and contiguous with
 * the shapes of kda_prefill_args; pinned (page-locked) host memory is needed
 * for the copies to overlap (pageable memory works but copies synchronously).
 * ws is a caller-owned device buffer of kda_prefill_host_workspace_size()
 * bytes, 256-byte aligned, holding the device copies of every tensor and the
 * prefill workspace; kda_prefill_device_status(ws) afterwards reports the
 * OR of the status words of all pieces.
 *
 * Ordering.  The copy streams first wait for work already queued on
 * `stream`; when `stream` reaches the point after this call, o and
 * final_state in host memory are complete.  The call creates and releases
 * its own CUDA events; it allocates no memory.  Snapshots and boundary
 * positions are not offered here (they live in device memory; use
 * kda_prefill).  cu_seqlens is validated on the host (cu[0] = 0,
 * non-decreasing, cu[N] = total_tokens): KDA_ERR_INVALID_ARG otherwise.
 */
typedef struct {
  int32_t num_seqs;            /* N >= 1                                          */
  int32_t num_heads;           /* H >= 1                                          */
  int32_t dk, dv;              /* each in {16, 32, 64, 128, 256}                  */
  int64_t total_tokens;        /* T = cu_seqlens[N]                               */
  const int64_t* cu_seqlens;   /* HOST [N+1]                                      */
  kda_dtype_t in_dtype;        /* dtype of q, k, v, g, b and of o                 */
  const void* q;               /* HOST [T, H, dk]                                 */
  const void* k;               /* HOST [T, H, dk]                                 */
  const void* v;               /* HOST [T, H, dv]                                 */
  const void* g;               /* HOST [T, H, dk]                                 */
  const void* b;               /* HOST [T, H]                                     */
  float scale;
  const float* initial_state;  /* HOST [N, H, dk, dv] or NULL (zeros)             */
  void* o;                     /* HOST [T, H, dv], in_dtype                       */
  float* final_state;          /* HOST [N, H, dk, dv] or NULL                     */
  int32_t segments;            /* pieces of the pipeline, 0 = default, <= 64     */
  void* copy_in_stream;        /* cudaStream_t for host->device copies (not `stream`) */
  void* copy_out_stream;       /* cudaStream_t for device->host copies (not `stream`) */
  int32_t gate_per_head;       /* as in kda_prefill_args: g is [T, H] when set    */
} kda_prefill_host_args;

/* Device workspace bytes kda_prefill_host needs (host-side fields only);
 * 0 if the arguments are invalid. */
size_t kda_prefill_host_workspace_size(const kda_prefill_host_args* args);

kda_status_t kda_prefill_host(const kda_prefill_host_args* args, void* ws, size_t ws_bytes,
                              void* stream);

/* Copies the workspace status word of the last kda_prefill that used `ws`
 * to *out (host), synchronising `stream`.  0 = clean; otherwise a bitwise OR
 * of 1 (malformed cu_seqlens), 2 (malformed boundary positions), 4 (chunk
 * table overflow), 8 (bounded wait expired), 16 (tensor-core path only: a
 * chunk's total decay in some key channel fell below 2^-250, about e^-173,
 * i.e. more than ~2.7 nats of log-decay per token on average over 64 tokens;
 * its operands leave the bf16 range and the results of such chunks are not
 * reliable -- fp32 inputs take the CUDA-core path, which has no such limit).
 * Below that bound the tensor-core path is exact in range: each channel's
 * decay factors are referred to half its chunk total. */
kda_status_t kda_prefill_device_status(const void* ws, int32_t* out, void* stream);

/* Host helper: snapshot slot offsets.  From host copies of cu_seqlens [n+1],
 * the interval and the boundary positions (may be NULL), fills
 * cu_snapshots_out [n+1] and returns the total number of snapshots, or -1 on
 * invalid input (boundaries not strictly increasing inside [1, len]). */
int64_t kda_snapshot_plan(const int64_t* h_cu_seqlens, int32_t n, int64_t interval,
                          const int64_t* h_boundary_pos, const int64_t* h_cu_boundaries,
                          int64_t* h_cu_snapshots_out);

/*
 * Snapshot retention (a prefix cache over a pool of saved states).
 *
 * A serving host keeps states of earlier prompts in a pool of device rows
 * ([rows, H, dk, dv] fp32, caller-owned) so that a later prompt sharing a
 * prefix resumes from the saved state instead of recomputing it ("Kimi K3:
 * The Manos, The Mythos, The Legendos", Context: the engine keeps selected
 * checkpoints, prompt boundaries among them; more of them cost memory and
 * save recomputation, so the retention policy matters).  These calls are
 * the policy: they track which row holds the state after which prefix of
 * token ids, and they never touch device memory.  They are the only calls of
 * the library that allocate (host memory for their index).
 *
 *   - An entry is keyed by its length p and two independent 64-bit hashes
 *     of the first p token ids (a false match needs both to collide).
 *   - kda_prefix_cache_lookup returns the longest cached prefix of
 *     tokens[0..n) (0 if none) and its row in *row (-1 if none), and marks
 *     it recently used.  Resume with initial_state = that row, over the
 *     tokens from p on.
 *   - kda_prefix_cache_reserve assigns rows for the states a prefill of
 *     tokens[0..n) will save at positions pos[0..m) (strictly increasing,
 *     1..n); is_boundary[i] != 0 marks prompt-boundary checkpoints (may be
 *     NULL: none).  rows_out[i] is the row to write, or -1 when the state
 *     is already cached (it is marked used) or no row could be freed.
 *     Pass rows_out as kda_prefill's snapshot_slot_map.  When the pool is
 *     full, interval checkpoints are evicted before boundary ones, least
 *     recently used first; boundary positions are placed first, then the
 *     others from the latest back, and a reservation never evicts a row it
 *     placed itself nor keep_row (the row the prefill resumes from, so that
 *     its initial state and its snapshots do not overlap; -1 = none).
 *     Returns the number of rows assigned, -1 on invalid arguments.  An
 *     entry is valid once the prefill that writes its row has run (order
 *     lookups' use of a row after it, e.g. on one stream).
 *   - A reserved entry is indexed at once.  If the prefill meant to write
 *     its rows fails (an error status, or a nonzero device status word), the
 *     caller must pass those rows to kda_prefix_cache_forget, which drops
 *     their entries and returns the rows to the free list, so that no later
 *     lookup resumes from a state that was never written.  Entries -1 (and
 *     rows not holding an entry) are ignored; returns the number of rows
 *     freed, -1 on invalid arguments (a row outside [-1, rows)).
 *   - Calls on one cache are serialised by an internal lock.
 */
typedef struct kda_prefix_cache kda_prefix_cache;

kda_prefix_cache* kda_prefix_cache_create(int64_t num_rows); /* NULL if num_rows < 1 */
void kda_prefix_cache_destroy(kda_prefix_cache* cache);
int64_t kda_prefix_cache_entries(kda_prefix_cache* cache);   /* -1 if cache is NULL */
int64_t kda_prefix_cache_lookup(kda_prefix_cache* cache, const int32_t* tokens, int64_t n,
                                int32_t* row);
int64_t kda_prefix_cache_reserve(kda_prefix_cache* cache, const int32_t* tokens, int64_t n,
                                 const int64_t* pos, const uint8_t* is_boundary, int64_t m,
                                 int32_t keep_row, int32_t* rows_out);
int64_t kda_prefix_cache_forget(kda_prefix_cache* cache, const int32_t* rows, int64_t m);

/*
 * One decode step for a batch of independent rows ("constant decode": a
 * single-token advance of each fixed-size state).  Row r advances the state
 * in pool slot state_slots[r] (slot r if state_slots is NULL; a negative
 * slot skips the row and leaves its o untouched) by its one token and
 * writes o.  The state is read once and written once, in place.
 */
typedef struct {
  int32_t batch;               /* B >= 0 rows                                     */
  int32_t num_heads;           /* H                                               */
  int32_t dk, dv;              /* each in {16, 32, 64, 128, 256}                  */
  int32_t num_slots;           /* rows of the state pool                          */
  kda_dtype_t in_dtype;        /* dtype of q, k, v, g, b and of o                 */
  float scale;
  const void* q;               /* device [B, H, dk]                               */
  const void* k;               /* device [B, H, dk]                               */
  const void* v;               /* device [B, H, dv]                               */
  const void* g;               /* device [B, H, dk]                               */
  const void* b;               /* device [B, H]                                   */
  float* state;                /* device pool [num_slots, H, dk, dv], in place    */
  const int32_t* state_slots;  /* device [B] or NULL; two rows must not share a slot */
  void* o;                     /* device [B, H, dv]                               */
  int64_t wait_limit_ns;       /* 0 = 1 s: the limit of the bounded waits of the
                                  128 x 128 kernel on its copies (see
                                  kda_prefill_args.wait_limit_ns)                 */
  int32_t* status;             /* device int32 or NULL: bit 8 is OR-ed in when a
                                  bounded wait gives up (the rows after it are
                                  then not updated)                               */
  int32_t gate_per_head;       /* as in kda_prefill_args: g is [B, H] when set    */
  const kda_layer_args* layer; /* host pointer, or NULL: the short convolution and
                                  output gate; windows [num_slots, conv_width - 1,
                                  H, d] indexed by the row's slot, updated in
                                  place when conv_out == conv_in.  The
                                  convolution needs dk * dv <= 128 * 128 here
                                  (KDA_ERR_UNSUPPORTED otherwise)               */
} kda_decode_args;

kda_status_t kda_decode_step(const kda_decode_args* args, void* stream);

/*
 * The preparation step on its own: for every token and head, q^ and k^
 * (L2-normalised), beta = sigmoid(b), and G, the running sum of
 * log alpha = -softplus(g) restarted at the start of each chunk of
 * KDA_CHUNK tokens of each sequence (chunks counted from the sequence
 * start).  kda_prefill performs the same step inside its intra-chunk kernel;
 * this entry exposes it.  Outputs are fp32: qhat, khat, G [T, H, dk];
 * beta [T, H].  Needs no workspace.
 */
typedef struct {
  int32_t num_seqs, num_heads, dk;
  int64_t total_tokens;
  const int64_t* cu_seqlens;   /* device [N+1]                                    */
  kda_dtype_t in_dtype;
  const void* q;
  const void* k;
  const void* g;
  const void* b;
  float* qhat;                 /* device [T, H, dk]                               */
  float* khat;                 /* device [T, H, dk]                               */
  float* G;                    /* device [T, H, dk]                               */
  float* beta;                 /* device [T, H]                                   */
  int32_t gate_per_head;       /* as in kda_prefill_args: g is [T, H] when set (G
                                  is still written [T, H, dk], equal across dk)  */
  const kda_layer_args* layer; /* host pointer, or NULL: with conv_width > 0, q
                                  and k pass through the short convolution
                                  before the normalisation, as in kda_prefill
                                  (conv_w[0..1], conv_in[0..1] used; windows
                                  [N, conv_width - 1, H, dk]; nothing else of
                                  the struct is read or written)               */
} kda_prep_args;

kda_status_t kda_prep(const kda_prep_args* args, void* stream);

/* Static description of a status code. */
const char* kda_status_string(kda_status_t status);

/* Library version string. */
const char* kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
