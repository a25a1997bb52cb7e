"""Independent numpy fp64 restatements of the KDA recurrence (pins for the oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing here shares
code with ``kda_oracle.c``; each function is written from the definition of
the recurrence and takes the gates directly:

    qhat, khat, alpha : [T, H, dk]    v : [T, H, dv]    beta : [T, H]

* ``product_form`` -- the update read literally as a product with an
  explicit transition matrix, S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
  + beta_t k_t v_t^T, o_t = scale S_t^T q_t.  The delta rule of "From KV Cache
  to Depth Attention" (Technical Details) with the diagonal gate of "Kimi K3:
  The Manos, The Mythos, The Legendos" (bullet list).
* ``brute_force_final`` -- the final state as the closed sum over tokens,
  S_T = A_T...A_1 S_0 + sum_s A_T...A_{s+1} beta_s k_s v_s^T with
  A_t = (I - beta_t k_t k_t^T) Diag(alpha_t); for tiny T and d.
* ``chunk_form`` -- the recurrence unrolled over chunks of C tokens (the
  "unrolling the recurrence in chunks" that "Kimi K3: The Manos, The Mythos,
  The Legendos" attributes to FlashKDA).  Within a chunk with start state
  S0 and cumulative decay Gamma_i = prod_{m<=i} alpha_m (per channel):
      A_kk[i,j] = beta_i sum_c k_ic k_jc Gamma_ic / Gamma_jc      (j < i)
      U         = (I + A_kk)^{-1} (diag(beta) V - diag(beta) (K o Gamma) S0)
      A_qk[i,j] = sum_c q_ic k_jc Gamma_ic / Gamma_jc            (j <= i)
      O         = scale ((Q o Gamma) S0 + A_qk U)
      S_end     = Diag(Gamma_L) S0 + (K o Gamma_L / Gamma)^T U
  derived by expanding the token recurrence inside the chunk; it is a design
  aid that must equal the token recurrence to rounding.
"""
from __future__ import annotations

import numpy as np


def product_form(qhat, khat, v, alpha, beta, scale=1.0, S0=None):
    """Token recurrence with explicit (I - beta k k^T) Diag(alpha) matrices."""
    T, H, dk = qhat.shape
    dv = v.shape[2]
    o = np.zeros((T, H, dv))
    S_all = np.zeros((H, dk, dv))
    for h in range(H):
        S = np.zeros((dk, dv)) if S0 is None else np.array(S0[h], dtype=np.float64)
        for t in range(T):
            k = khat[t, h][:, None]
            A = (np.eye(dk) - beta[t, h] * (k @ k.T)) @ np.diag(alpha[t, h])
            S = A @ S + beta[t, h] * (k @ v[t, h][None, :])
            o[t, h] = scale * (S.T @ qhat[t, h])
        S_all[h] = S
    return o, S_all


def brute_force_final(khat, v, alpha, beta, S0=None):
    """Final state as a sum over tokens of transported rank-1 writes."""
    T, H, dk = khat.shape
    dv = v.shape[2]
    out = np.zeros((H, dk, dv))
    for h in range(H):
        A = []
        for t in range(T):
            k = khat[t, h][:, None]
            A.append((np.eye(dk) - beta[t, h] * (k @ k.T)) @ np.diag(alpha[t, h]))

        def transport(a, b):  # A_b ... A_a (identity when a > b)
            P = np.eye(dk)
            for t in range(a, b + 1):
                P = A[t] @ P
            return P

        S = np.zeros((dk, dv))
        if S0 is not None:
            S += transport(0, T - 1) @ S0[h]
        for s in range(T):
            S += transport(s + 1, T - 1) @ (beta[s, h] * np.outer(khat[s, h], v[s, h]))
        out[h] = S
    return out


def chunk_form(qhat, khat, v, log_alpha, beta, scale=1.0, S0=None, C=64):
    """Chunked evaluation; chunks of C tokens with a ragged last chunk."""
    T, H, dk = qhat.shape
    dv = v.shape[2]
    o = np.zeros((T, H, dv))
    S_all = np.zeros((H, dk, dv))
    for h in range(H):
        S = np.zeros((dk, dv)) if S0 is None else np.array(S0[h], dtype=np.float64)
        for c0 in range(0, T, C):
            c1 = min(c0 + C, T)
            Q = qhat[c0:c1, h]; K = khat[c0:c1, h]; V = v[c0:c1, h]
            bt = beta[c0:c1, h]
            G = np.cumsum(log_alpha[c0:c1, h], axis=0)       # log Gamma_i, [L, dk]
            L = c1 - c0
            ratio = np.exp(G[:, None, :] - G[None, :, :])       # Gamma_i / Gamma_j, [L, L, dk]
            Kraw = np.einsum("ic,jc,ijc->ij", K, K, ratio)
            Akk = np.tril(bt[:, None] * Kraw, k=-1)
            Aqk = np.tril(np.einsum("ic,jc,ijc->ij", Q, K, ratio), k=0)
            Tinv = np.linalg.inv(np.eye(L) + Akk)
            KG = K * np.exp(G)
            U = Tinv @ (bt[:, None] * V - bt[:, None] * (KG @ S))
            o[c0:c1, h] = scale * ((Q * np.exp(G)) @ S + Aqk @ U)
            GL = G[-1]
            S = np.exp(GL)[:, None] * S + (K * np.exp(GL[None, :] - G)).T @ U
        S_all[h] = S
    return o, S_all
