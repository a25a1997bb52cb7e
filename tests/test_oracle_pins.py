"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

No test here retypes the oracle's formula: each compares it with a closed
form, an exact special case, a hand-worked example, brute force, an
independent numpy restatement (product form / chunk form), autograd, or an
invariant.  CPU only.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import forms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed):
    return np.random.default_rng(seed)


def random_inputs(rng, T, H, dk, dv, g_mean=-3.0):
    q = rng.standard_normal((T, H, dk)).astype(np.float32)
    k = rng.standard_normal((T, H, dk)).astype(np.float32)
    v = rng.standard_normal((T, H, dv)).astype(np.float32)
    g = (rng.standard_normal((T, H, dk)) + g_mean).astype(np.float32)
    b = rng.standard_normal((T, H)).astype(np.float32)
    return q, k, v, g, b


def gates(oracle_mod, q, k, g, b):
    qh, kh, la, be = oracle_mod.prep(q, k, g, b)
    return qh, kh, np.exp(la), la, be


# ---------------------------------------------------------------- prep closed forms
def test_prep_closed_forms(oracle_mod):
    q = np.array([[3.0, 4.0, 0.0], [0.0, 0.0, 0.0], [1e-8, 0.0, 0.0]], np.float32)
    k = np.array([[0.0, 0.0, 2.0], [1.0, 0.0, 0.0], [0.0, -5.0, 0.0]], np.float32)
    g = np.array([[0.0, math.log(math.e - 1.0), -1e30],
                  [30.0, -40.0, 5.0], [-3.0, 1.0, -1.0]], np.float32)
    b = np.array([0.0, math.log(3.0), -1e30], np.float32)
    qh, kh, la, be = oracle_mod.prep(q, k, g, b)
    np.testing.assert_allclose(qh[0], [0.6, 0.8, 0.0], rtol=0, atol=1e-15)
    assert np.all(qh[1] == 0.0)                                   # zero vector stays 0
    np.testing.assert_allclose(qh[2], [float(np.float32(1e-8)) / 1e-6, 0, 0], rtol=1e-15)  # norm floor
    np.testing.assert_allclose(kh[0], [0, 0, 1.0], atol=0)
    np.testing.assert_allclose(kh[2], [0, -1.0, 0], atol=0)
    # log alpha = -softplus(g): softplus(0)=log 2, softplus(log(e-1)) = 1, softplus(-inf)=0
    np.testing.assert_allclose(la[0], [-math.log(2.0), -1.0, 0.0], rtol=1e-7, atol=0)
    assert la[0, 2] == 0.0                                        # alpha exactly 1
    np.testing.assert_allclose(la[1, 0], -30.0 - math.log1p(math.exp(-30.0)), rtol=1e-12)
    np.testing.assert_allclose(la[1, 1], -math.log1p(math.exp(-40.0)), rtol=1e-12)
    np.testing.assert_allclose(la[1, 2], -math.log1p(math.exp(5.0)), rtol=1e-14)
    # beta = sigmoid(b): sigmoid(0)=1/2, sigmoid(log 3) = 3/4, sigmoid(-inf) = 0
    np.testing.assert_allclose(be, [0.5, 0.75, 0.0], rtol=1e-7, atol=0)
    assert be[2] == 0.0


# ---------------------------------------------------------------- hand-worked example
def test_golden_worked_example(oracle_mod):
    with open(os.path.join(GOLDEN, "kda_tiny_worked.json")) as f:
        gold = json.load(f)
    inp = {key: np.array(val, dtype=np.float32) for key, val in gold["inputs"].items()}
    o, S, _ = oracle_mod.prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], [0, 2])
    tol = gold["tolerance_abs"]
    np.testing.assert_allclose(o, np.array(gold["expected"]["o"]), rtol=0, atol=tol)
    np.testing.assert_allclose(S[0], np.array(gold["expected"]["S_final"]), rtol=0, atol=tol)


# ---------------------------------------------------------------- exact retrieval
@pytest.mark.parametrize("dk", [8, 16])
def test_orthonormal_retrieval_exact(oracle_mod, dk):
    """Orthonormal keys, alpha = 1, beta = 1, zero state: a query equal to an
    earlier key returns that key's value bit for bit (lookup by address)."""
    rng = rnd(1)
    T, dv = dk, 5
    perm = rng.permutation(dk)
    k = np.zeros((T, 1, dk), np.float32)
    k[np.arange(T), 0, perm[:T]] = 1.0
    target = np.array([rng.integers(0, t + 1) for t in range(T)])
    q = k[target].copy()
    v = rng.standard_normal((T, 1, dv)).astype(np.float32)
    g = np.full((T, 1, dk), -1e30, np.float32)        # alpha = 1 exactly
    b = np.full((T, 1), 100.0, np.float32)            # beta = 1 exactly
    o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T])
    assert np.array_equal(o[:, 0], v[target, 0].astype(np.float64))
    # the state is the sum of the stored outer products, exactly
    expect = np.zeros((dk, dv))
    for t in range(T):
        expect[perm[t]] += v[t, 0]
    assert np.array_equal(S[0, 0], expect)


def test_delta_overwrite_invariant(oracle_mod):
    """After a token, S_t^T k_t = (1 - beta) S'^T k_t + beta v_t; with beta = 1
    the state returns v_t exactly for its own key whatever the history."""
    rng = rnd(2)
    T, H, dk, dv = 24, 2, 8, 6
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    b[::2] = 100.0                                     # beta = 1 on even tokens
    pos = np.arange(1, T + 1)
    o, S, snaps = oracle_mod.prefill(q, k, v, g, b, [0, T], snap_pos=pos, cu_snap=[0, T])
    qh, kh, alpha, _, be = gates(oracle_mod, q, k, g, b)
    prev = np.zeros((H, dk, dv))
    for t in range(T):
        for h in range(H):
            Sp = alpha[t, h][:, None] * prev[h]
            lhs = snaps[t, h].T @ kh[t, h]
            rhs = (1 - be[t, h]) * (Sp.T @ kh[t, h]) + be[t, h] * v[t, h]
            np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
            if t % 2 == 0:
                np.testing.assert_allclose(lhs, v[t, h], rtol=0, atol=1e-12)
        prev = snaps[t]


def test_beta_zero_pure_decay(oracle_mod):
    """beta = 0: the update is pure per-channel decay of the initial state."""
    rng = rnd(3)
    T, H, dk, dv = 30, 2, 8, 4
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv, g_mean=-1.0)
    b[:] = -1e30                                       # beta = 0 exactly
    S0 = rng.standard_normal((1, H, dk, dv))
    o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], scale=0.5, S0=S0)
    la = -np.logaddexp(0.0, g.astype(np.float64))      # log alpha, closed form of softplus
    cum = np.cumsum(la, axis=0)                        # log prod_{m<=t} alpha_m
    qn = q / np.linalg.norm(q.astype(np.float64), axis=-1, keepdims=True)
    for h in range(H):
        np.testing.assert_allclose(S[0, h], np.exp(cum[-1, h])[:, None] * S0[0, h],
                                   rtol=1e-12, atol=0)
        for t in range(T):
            expect = 0.5 * (np.exp(cum[t, h])[:, None] * S0[0, h]).T @ qn[t, h]
            np.testing.assert_allclose(o[t, h], expect, rtol=1e-12, atol=1e-14)


def test_order_sensitivity(oracle_mod):
    """Reversing the tokens changes the state for generic inputs; for
    orthonormal keys with alpha = 1 the writes commute and it does not."""
    rng = rnd(4)
    T, H, dk, dv = 16, 1, 8, 8
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    _, S_fwd, _ = oracle_mod.prefill(q, k, v, g, b, [0, T])
    _, S_rev, _ = oracle_mod.prefill(q[::-1], k[::-1], v[::-1], g[::-1], b[::-1], [0, T])
    assert np.linalg.norm(S_fwd - S_rev) > 1e-2 * np.linalg.norm(S_fwd)
    k2 = np.zeros((dk, 1, dk), np.float32)
    k2[np.arange(dk), 0, rng.permutation(dk)] = 1.0
    q2, v2 = q[:dk], v[:dk]
    g2 = np.full((dk, 1, dk), -1e30, np.float32)
    b2 = rng.standard_normal((dk, 1)).astype(np.float32)
    _, A, _ = oracle_mod.prefill(q2, k2, v2, g2, b2, [0, dk])
    _, B, _ = oracle_mod.prefill(q2[::-1], k2[::-1], v2[::-1], g2[::-1], b2[::-1], [0, dk])
    np.testing.assert_allclose(A, B, rtol=0, atol=1e-15)


# ---------------------------------------------------------------- independent forms
@pytest.mark.parametrize("T,dk,dv", [(1, 1, 1), (5, 3, 2), (8, 4, 4)])
def test_brute_force_expansion(oracle_mod, T, dk, dv):
    rng = rnd(10 + T)
    H = 2
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv, g_mean=-0.5)
    S0 = rng.standard_normal((1, H, dk, dv))
    _, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], S0=S0)
    qh, kh, alpha, _, be = gates(oracle_mod, q, k, g, b)
    S_bf = forms.brute_force_final(kh, v.astype(np.float64), alpha, be, S0=S0[0])
    np.testing.assert_allclose(S[0], S_bf, rtol=0, atol=1e-13)


def test_product_form_and_recurrence_core(oracle_mod):
    """The delta form (oracle) equals the literal product form; the gate-level
    core equals the prefill entry on the same gates."""
    rng = rnd(20)
    T, H, dk, dv = 40, 3, 8, 6
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.3
    o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], scale=0.75, S0=S0)
    qh, kh, alpha, _, be = gates(oracle_mod, q, k, g, b)
    o_p, S_p = forms.product_form(qh, kh, v.astype(np.float64), alpha, be, 0.75, S0[0])
    np.testing.assert_allclose(o, o_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S[0], S_p, rtol=0, atol=1e-12)
    o_c, S_c = oracle_mod.recurrence(qh, kh, v, alpha, be, 0.75, S0[0])
    np.testing.assert_allclose(o_c, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S_c, S[0], rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", ["gated_scalar", "deltanet"])
def test_special_cases(oracle_mod, case):
    """alpha equal across channels = gated delta rule; alpha = 1 = DeltaNet
    ("Kimi K3: The Manos, The Mythos, The Legendos", bullet list)."""
    rng = rnd(30)
    T, H, dk, dv = 32, 2, 8, 8
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    if case == "gated_scalar":
        g[:] = g[:, :, :1]
    else:
        g[:] = -1e30
    o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T])
    qh, kh, alpha, _, be = gates(oracle_mod, q, k, g, b)
    if case == "deltanet":
        assert np.all(alpha == 1.0)
    else:
        assert np.all(alpha == alpha[:, :, :1])
    o_p, S_p = forms.product_form(qh, kh, v.astype(np.float64), alpha, be)
    np.testing.assert_allclose(o, o_p, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S[0], S_p, rtol=0, atol=1e-12)


def test_online_learning_gradient_step(oracle_mod):
    """Each token is one gradient step of size beta on 1/2 |S'^T k - v|^2,
    taken at S' = Diag(alpha) S_{t-1} (gradient from torch autograd)."""
    torch = pytest.importorskip("torch")
    rng = rnd(40)
    T, H, dk, dv = 6, 1, 5, 4
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    pos = np.arange(1, T + 1)
    _, _, snaps = oracle_mod.prefill(q, k, v, g, b, [0, T], snap_pos=pos, cu_snap=[0, T])
    _, kh, alpha, _, be = gates(oracle_mod, q, k, g, b)
    prev = np.zeros((dk, dv))
    for t in range(T):
        Sp = torch.tensor(alpha[t, 0][:, None] * prev, requires_grad=True)
        kt = torch.tensor(kh[t, 0]); vt = torch.tensor(v[t, 0].astype(np.float64))
        loss = 0.5 * ((Sp.T @ kt - vt) ** 2).sum()
        loss.backward()
        step = (Sp - be[t, 0] * Sp.grad).detach().numpy()
        np.testing.assert_allclose(snaps[t, 0], step, rtol=0, atol=1e-13)
        prev = snaps[t, 0]


def test_contraction_bound(oracle_mod):
    """With 0 <= beta <= 1, alpha <= 1 and unit keys the transition is a
    contraction: |S_t|_2 <= |S_{t-1}|_2 + beta_t |v_t|."""
    rng = rnd(50)
    T, H, dk, dv = 64, 2, 16, 16
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv, g_mean=-1.0)
    pos = np.arange(1, T + 1)
    S0 = rng.standard_normal((1, H, dk, dv))
    _, _, snaps = oracle_mod.prefill(q, k, v, g, b, [0, T], S0=S0, snap_pos=pos,
                                     cu_snap=[0, T])
    _, _, _, _, be = gates(oracle_mod, q, k, g, b)
    prev = S0[0]
    for t in range(T):
        for h in range(H):
            lhs = np.linalg.norm(snaps[t, h], 2)
            rhs = np.linalg.norm(prev[h], 2) + be[t, h] * np.linalg.norm(v[t, h].astype(float))
            assert lhs <= rhs * (1 + 1e-12)
        prev = snaps[t]


@pytest.mark.parametrize("C", [16, 64])
def test_chunk_form_equivalence(oracle_mod, C):
    """The chunked algebra equals the token recurrence (ragged last chunk)."""
    rng = rnd(60 + C)
    T, H, dk, dv = 150, 2, 16, 12
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((1, H, dk, dv)) * 0.1
    o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], scale=0.9, S0=S0)
    qh, kh, _, la, be = gates(oracle_mod, q, k, g, b)
    o_c, S_c = forms.chunk_form(qh, kh, v.astype(np.float64), la, be, 0.9, S0[0], C=C)
    np.testing.assert_allclose(o_c, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_c, S[0], rtol=0, atol=1e-12)


def test_state_map_is_affine(oracle_mod):
    """The recurrence is affine in the state: over any run of tokens,
    S_end = A S_start + B with A the run from the identity with v = 0 and B
    the run from zero -- the property the segment scan relies on.  Checked on
    a random start state and on a split into two runs composed by hand."""
    rng = rnd(65)
    T, H, d = 90, 2, 8
    q, k, v, g, b = random_inputs(rng, T, H, d, d)
    eye = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    zero_v = np.zeros_like(v)
    _, A, _ = oracle_mod.prefill(q, k, zero_v, g, b, [0, T], S0=eye)
    _, B, _ = oracle_mod.prefill(q, k, v, g, b, [0, T])
    S0 = rng.standard_normal((1, H, d, d))
    _, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], S0=S0)
    np.testing.assert_allclose(S[0], np.einsum("hij,hjk->hik", A[0], S0[0]) + B[0], rtol=0, atol=1e-12)
    # two runs: S_end = A2 (A1 S0 + B1) + B2
    p = 41
    _, A1, _ = oracle_mod.prefill(q[:p], k[:p], zero_v[:p], g[:p], b[:p], [0, p], S0=eye)
    _, B1, _ = oracle_mod.prefill(q[:p], k[:p], v[:p], g[:p], b[:p], [0, p])
    _, A2, _ = oracle_mod.prefill(q[p:], k[p:], zero_v[p:], g[p:], b[p:], [0, T - p], S0=eye)
    _, B2, _ = oracle_mod.prefill(q[p:], k[p:], v[p:], g[p:], b[p:], [0, T - p])
    mid = np.einsum("hij,hjk->hik", A1[0], S0[0]) + B1[0]
    np.testing.assert_allclose(np.einsum("hij,hjk->hik", A2[0], mid) + B2[0], S[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------- serving semantics
def test_resume_from_snapshot(oracle_mod):
    """Prefill of [0,p) then of [p,len) from the state at p equals one pass
    (snapshot reuse, "Kimi K3: The Manos, The Mythos, The Legendos", Context)."""
    rng = rnd(70)
    T, H, dk, dv, p = 100, 2, 8, 8, 37
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    o, S, snaps = oracle_mod.prefill(q, k, v, g, b, [0, T], snap_pos=[p], cu_snap=[0, 1])
    o1, S1, _ = oracle_mod.prefill(q[:p], k[:p], v[:p], g[:p], b[:p], [0, p])
    np.testing.assert_allclose(S1, snaps[:1], rtol=0, atol=0)
    o2, S2, _ = oracle_mod.prefill(q[p:], k[p:], v[p:], g[p:], b[p:], [0, T - p], S0=S1)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(S2, S, rtol=0, atol=1e-13)


def test_varlen_packing_and_snapshots(oracle_mod):
    """Packed sequences are independent; snapshot slots follow the sorted
    union of interval multiples and boundary positions."""
    rng = rnd(80)
    lens = [5, 70, 1, 33]
    H, dk, dv = 2, 8, 4
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, b = random_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv)) * 0.1
    bpos = np.array([3, 5, 10, 64, 70, 1, 33], np.int64)
    cub = np.array([0, 2, 5, 6, 7], np.int64)
    sp, cs = oracle_mod.snapshot_positions(lens, 32, bpos, cub)
    assert list(sp) == [3, 5, 10, 32, 64, 70, 1, 32, 33]
    assert list(cs) == [0, 2, 6, 7, 9]
    o, S, snaps = oracle_mod.prefill(q, k, v, g, b, cu, S0=S0, snap_pos=sp, cu_snap=cs)
    for s, L in enumerate(lens):
        a, e = cu[s], cu[s + 1]
        o_s, S_s, _ = oracle_mod.prefill(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], [0, L],
                                         S0=S0[s:s + 1])
        np.testing.assert_allclose(o[a:e], o_s, rtol=0, atol=0)
        np.testing.assert_allclose(S[s], S_s[0], rtol=0, atol=0)
        for j in range(cs[s], cs[s + 1]):
            p = sp[j]
            _, S_p, _ = oracle_mod.prefill(q[a:a + p], k[a:a + p], v[a:a + p], g[a:a + p],
                                           b[a:a + p], [0, p], S0=S0[s:s + 1])
            np.testing.assert_allclose(snaps[j], S_p[0], rtol=0, atol=0)


def test_decode_equals_prefill(oracle_mod):
    """T decode steps from a state equal a T-token prefill from that state;
    slot indirection permutes rows and a negative slot skips a row."""
    rng = rnd(90)
    B, H, dk, dv, T = 3, 2, 8, 8, 12
    S0 = rng.standard_normal((B, H, dk, dv)) * 0.1
    steps = [random_inputs(rng, B, H, dk, dv) for _ in range(T)]
    state = S0.copy()
    outs = [oracle_mod.decode(*st, state) for st in steps]
    for r in range(B):
        q = np.stack([st[0][r] for st in steps]); k = np.stack([st[1][r] for st in steps])
        v = np.stack([st[2][r] for st in steps]); g = np.stack([st[3][r] for st in steps])
        b = np.stack([st[4][r] for st in steps])
        o, S, _ = oracle_mod.prefill(q, k, v, g, b, [0, T], S0=S0[r:r + 1])
        np.testing.assert_allclose(np.stack([ot[r] for ot in outs]), o, rtol=0, atol=1e-14)
        np.testing.assert_allclose(state[r], S[0], rtol=0, atol=1e-14)
    pool = S0.copy()
    slots = np.array([2, -1, 0], np.int32)
    o = oracle_mod.decode(*steps[0], pool, slots=slots)
    assert np.all(o[1] == 0.0)
    np.testing.assert_array_equal(pool[1], S0[1])
    st0 = steps[0]
    one = S0[[2]].copy()
    o_a = oracle_mod.decode(st0[0][[0]], st0[1][[0]], st0[2][[0]], st0[3][[0]], st0[4][[0]], one)
    np.testing.assert_array_equal(o[0], o_a[0])
    np.testing.assert_array_equal(pool[2], one[0])
