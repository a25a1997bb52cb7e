/*
 * kda_oracle.c -- plain, slow, fp64 CPU oracle of the Kimi Delta Attention
 * (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code,
 * header, table or helper with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it computes (one head, one sequence, token by token):
 *
 *   q^ = q / max(|q|, 1e-6)          k^ = k / max(|k|, 1e-6)
 *   beta = sigmoid(b)                alpha_c = exp(-softplus(g_c))
 *   S'  = Diag(alpha) S              retention of the old state
 *   p   = S'^T k^                    the state first predicts the value
 *   S   = S' + beta k^ (v - p)^T     and writes back only the difference
 *   o   = scale * S^T q^             read-out with the updated state
 *
 * which is algebraically the product form
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T.
 *
 * Sources:
 *  - "From KV Cache to Depth Attention: The Bottlenecks Kimi K3 Had to
 *    Break", section Technical Details, bullet "Kimi Delta Attention (KDA)":
 *    predict from the existing memory, write only the delta; alpha is the
 *    retention, beta the update strength; each feature channel has its own
 *    timescale (hence a per-channel alpha, i.e. a diagonal gate).
 *  - "Kimi K3: The Manos, The Mythos, The Legendos", bullet list: linear
 *    attention -> delta rule -> forget gate -> the gate made a diagonal
 *    matrix; queries and keys are L2-normalised (stability bullet).
 *  - Same page, section Context: the engine keeps state snapshots at chosen
 *    positions (prompt boundaries) for later reuse -> the snapshot outputs.
 *
 * Readings where the pages are silent: the L2-norm floor 1e-6, beta as a
 * sigmoid of a per-(token, head) logit b, alpha = exp(-softplus(g)) per
 * channel, and o read from the state after the token's own update.
 *
 * Layouts (all row-major, token-major packed like the GPU library):
 *   q, k, g : [T_total, H, dk]     v : [T_total, H, dv]     b : [T_total, H]
 *   states  : [.., H, dk, dv]      o : [T_total, H, dv]
 * Inputs are float32 (bf16 inputs are passed as their exact float32 values);
 * all arithmetic and all outputs are double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x); for x > 20 the correction log1p(e^-x) is below
 * double's resolution of x, so x itself is returned. */
static double oracle_softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

static double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* x^ = x / max(|x|, 1e-6).  A unit vector is returned unchanged (exactly). */
static void oracle_l2norm(const float* x, int n, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  double nrm = sqrt(ss);
  if (nrm < 1e-6) nrm = 1e-6;
  for (int i = 0; i < n; ++i) out[i] = (double)x[i] / nrm;
}

/* One token of the recurrence on state S [dk, dv], in place.
 * alpha [dk], khat [dk], qhat [dk] (may be NULL: no read-out), v [dv].
 * p and u are scratch of length dv.  o (length dv) receives scale*S^T qhat. */
static void oracle_token_step(int dk, int dv, double* S, const double* alpha,
                              const double* khat, const double* qhat,
                              const double* v, double beta, double scale,
                              double* p, double* u, double* o) {
  /* retention: S' = Diag(alpha) S (row c of S is channel c of the key) */
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] *= alpha[c];
  /* prediction from the existing memory: p = S'^T k^ */
  for (int j = 0; j < dv; ++j) p[j] = 0.0;
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) p[j] += S[(size_t)c * dv + j] * khat[c];
  /* only the difference is written: S = S' + beta k^ (v - p)^T */
  for (int j = 0; j < dv; ++j) u[j] = beta * (v[j] - p[j]);
  for (int c = 0; c < dk; ++c)
    for (int j = 0; j < dv; ++j) S[(size_t)c * dv + j] += khat[c] * u[j];
  /* read-out with the updated state: o = scale * S^T q^ */
  if (qhat && o) {
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int c = 0; c < dk; ++c)
      for (int j = 0; j < dv; ++j) o[j] += S[(size_t)c * dv + j] * qhat[c];
    for (int j = 0; j < dv; ++j) o[j] *= scale;
  }
}

/* Per-token preparation of one (token, head): normalised q and k, the
 * per-channel log-retention log(alpha) = -softplus(g) and beta = sigmoid(b).
 * Exposed so that its closed forms can be checked on their own. */
void kda_oracle_prep(int64_t n_rows, int32_t dk, const float* q, const float* k,
                     const float* g, const float* b, double* qhat, double* khat,
                     double* log_alpha, double* beta) {
  for (int64_t r = 0; r < n_rows; ++r) {
    oracle_l2norm(q + r * dk, dk, qhat + r * dk);
    oracle_l2norm(k + r * dk, dk, khat + r * dk);
    for (int c = 0; c < dk; ++c)
      log_alpha[r * dk + c] = -oracle_softplus((double)g[r * dk + c]);
    beta[r] = oracle_sigmoid((double)b[r]);
  }
}

static int oracle_threads(int32_t nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/*
 * Prefill over packed variable-length sequences.
 *   cu_seqlens [N+1]: sequence s holds packed tokens [cu[s], cu[s+1]).
 *   S0 [N, H, dk, dv] or NULL (zero initial state).
 *   o [T_total, H, dv], S_final [N, H, dk, dv] (may be NULL).
 *   Snapshots: snap_pos holds, for sequence s, the sorted seq-relative
 *   positions snap_pos[cu_snap[s] .. cu_snap[s+1]); the state after that many
 *   tokens of the sequence is written to snaps[slot, h] with slot the same
 *   index.  snap_pos/cu_snap/snaps may be NULL.
 *   Only heads in [h_begin, h_end) are computed; other outputs are untouched.
 * Returns 0, or -1 on an inconsistent argument.
 */
int kda_oracle_prefill(int32_t N, int32_t H, int32_t dk, int32_t dv,
                       const int64_t* cu_seqlens, const float* q,
                       const float* k, const float* v, const float* g,
                       const float* b, double scale, const double* S0,
                       double* o, double* S_final, const int64_t* snap_pos,
                       const int64_t* cu_snap, double* snaps, int32_t h_begin,
                       int32_t h_end, int32_t nthreads) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  if (h_begin < 0 || h_end > H || h_begin > h_end) return -1;
  for (int32_t s = 0; s < N; ++s)
    if (cu_seqlens[s + 1] < cu_seqlens[s]) return -1;
  const int64_t n_pairs = (int64_t)N * (h_end - h_begin);
  const size_t sz = (size_t)dk * dv;
  int bad = 0;

#pragma omp parallel num_threads(oracle_threads(nthreads)) reduction(| : bad)
  {
    double* S = (double*)malloc(sizeof(double) * sz);
    double* work = (double*)malloc(sizeof(double) * (3 * (size_t)dk + 4 * (size_t)dv + 1));
    double* qh = work;
    double* kh = qh + dk;
    double* al = kh + dk;
    double* vv = al + dk;
    double* p = vv + dv;
    double* u = p + dv;
    double* ot = u + dv;
#pragma omp for schedule(dynamic, 1)
    for (int64_t pair = 0; pair < n_pairs; ++pair) {
      const int32_t s = (int32_t)(pair / (h_end - h_begin));
      const int32_t h = h_begin + (int32_t)(pair % (h_end - h_begin));
      const int64_t t0 = cu_seqlens[s], len = cu_seqlens[s + 1] - cu_seqlens[s];
      if (S0)
        memcpy(S, S0 + ((size_t)s * H + h) * sz, sizeof(double) * sz);
      else
        memset(S, 0, sizeof(double) * sz);
      int64_t snap_i = 0, snap_n = 0, snap_base = 0;
      if (snap_pos && cu_snap && snaps) {
        snap_base = cu_snap[s];
        snap_n = cu_snap[s + 1] - cu_snap[s];
      }
      for (int64_t t = 0; t < len; ++t) {
        const int64_t row = (t0 + t) * H + h;
        oracle_l2norm(q + row * dk, dk, qh);
        oracle_l2norm(k + row * dk, dk, kh);
        for (int c = 0; c < dk; ++c)
          al[c] = exp(-oracle_softplus((double)g[row * dk + c]));
        for (int j = 0; j < dv; ++j) vv[j] = (double)v[row * dv + j];
        const double beta = oracle_sigmoid((double)b[row]);
        oracle_token_step(dk, dv, S, al, kh, qh, vv, beta, scale, p, u, ot);
        for (int j = 0; j < dv; ++j) o[row * dv + j] = ot[j];
        while (snap_i < snap_n && snap_pos[snap_base + snap_i] == t + 1) {
          memcpy(snaps + ((size_t)(snap_base + snap_i) * H + h) * sz, S,
                 sizeof(double) * sz);
          ++snap_i;
        }
      }
      if (snap_i != snap_n) bad = 1; /* a position outside [1, len] or unsorted */
      if (S_final) memcpy(S_final + ((size_t)s * H + h) * sz, S, sizeof(double) * sz);
    }
    free(work);
    free(S);
  }
  return bad ? -1 : 0;
}

/*
 * The recurrence core with the gates given directly (no preparation step):
 * qhat, khat, alpha [T, H, dk] and beta [T, H] as doubles, v [T, H, dv].
 * Used by the property checks that need alpha or beta exactly 0 or 1.
 * One sequence of T tokens; S0/S_final [H, dk, dv]; o [T, H, dv].
 */
void kda_oracle_recurrence(int64_t T, int32_t H, int32_t dk, int32_t dv,
                           const double* qhat, const double* khat,
                           const double* v, const double* alpha,
                           const double* beta, double scale, const double* S0,
                           double* o, double* S_final) {
  const size_t sz = (size_t)dk * dv;
  double* S = (double*)malloc(sizeof(double) * sz);
  double* p = (double*)malloc(sizeof(double) * 2 * (size_t)dv);
  double* u = p + dv;
  for (int32_t h = 0; h < H; ++h) {
    if (S0)
      memcpy(S, S0 + (size_t)h * sz, sizeof(double) * sz);
    else
      memset(S, 0, sizeof(double) * sz);
    for (int64_t t = 0; t < T; ++t) {
      const int64_t row = t * H + h;
      oracle_token_step(dk, dv, S, alpha + row * dk, khat + row * dk,
                        qhat + row * dk, v + row * dv, beta[row], scale, p, u,
                        o + row * dv);
    }
    if (S_final) memcpy(S_final + (size_t)h * sz, S, sizeof(double) * sz);
  }
  free(p);
  free(S);
}

/*
 * One decode step for a batch of B independent rows: row r advances the
 * state held in pool slot slots[r] (slots NULL: slot r; slot < 0: the row is
 * skipped and its o is left untouched) by one token.
 *   q, k, g [B, H, dk], v [B, H, dv], b [B, H] float32;
 *   state [n_slots, H, dk, dv] double, updated in place; o [B, H, dv].
 * The step is the same token update as the prefill: "constant decode" in
 * "Kimi K3: The Manos, The Mythos, The Legendos" (bullet on FlashKDA) is this
 * one-token advance of a fixed-size state.
 */
void kda_oracle_decode(int32_t B, int32_t H, int32_t dk, int32_t dv,
                       const float* q, const float* k, const float* v,
                       const float* g, const float* b, double scale,
                       double* state, const int32_t* slots, double* o,
                       int32_t nthreads) {
  const size_t sz = (size_t)dk * dv;
  const int64_t n_pairs = (int64_t)B * H;
#pragma omp parallel num_threads(oracle_threads(nthreads))
  {
    double* work = (double*)malloc(sizeof(double) * (3 * (size_t)dk + 4 * (size_t)dv));
    double* qh = work;
    double* kh = qh + dk;
    double* al = kh + dk;
    double* vv = al + dk;
    double* p = vv + dv;
    double* u = p + dv;
    double* ot = u + dv;
#pragma omp for schedule(static)
    for (int64_t pair = 0; pair < n_pairs; ++pair) {
      const int32_t r = (int32_t)(pair / H), h = (int32_t)(pair % H);
      const int32_t slot = slots ? slots[r] : r;
      if (slot < 0) continue;
      const int64_t row = (int64_t)r * H + h;
      oracle_l2norm(q + row * dk, dk, qh);
      oracle_l2norm(k + row * dk, dk, kh);
      for (int c = 0; c < dk; ++c) al[c] = exp(-oracle_softplus((double)g[row * dk + c]));
      for (int j = 0; j < dv; ++j) vv[j] = (double)v[row * dv + j];
      const double beta = oracle_sigmoid((double)b[row]);
      oracle_token_step(dk, dv, state + ((size_t)slot * H + h) * sz, al, kh, qh,
                        vv, beta, scale, p, u, ot);
      for (int j = 0; j < dv; ++j) o[row * dv + j] = ot[j];
    }
    free(work);
  }
}

int kda_oracle_max_threads(void) { return oracle_threads(0); }
