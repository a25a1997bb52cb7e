"""The method's exact special cases through the CUDA path (tensor-core
prefill, bf16, 128 x 128 heads, and the decode ring kernel), against the
oracle and against what the recurrence gives in closed form.

* alpha = 1 exactly (g = -60: the delta rule without decay, "Kimi K3: The
  Manos, The Mythos, The Legendos", bullet list -- DeltaNet before the gate);
* beta = 0 exactly (b = -100): no write, the state only decays, so
  S_T = Diag(prod alpha) S_0 and o_t = scale (Diag(Gamma_t) S_0)^T q^_t;
* beta = 1 exactly (b = +100) with q = k: the delta rule overwrites the value
  stored under k^ ("From KV Cache to Depth Attention", Technical Details:
  predict, then write the difference), so o_t = S_t^T k^_t = v_t;
* zero q or k rows (the norm floor maps them to zero vectors): o = 0 exactly
  for q = 0, and a k = 0 token writes nothing;
* orthonormal retrieval at dk = 128 with alpha = beta = 1: 128 keys e_pi(t)
  store v_t, later queries e_pi(j) read v_j back, and the state holds v_t
  in row pi(t).

Tolerances: 5e-3 relative Frobenius error against the oracle (bf16 inputs),
as in the other parity tests; the closed forms that involve no rounding in
the kernels' arithmetic (retrieval, q = 0) are checked to 1e-6 or exactly.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_delta_gb300 import kda
from linear_attention_serving_delta_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 5e-3


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def host(t):
    return t.detach().float().cpu().numpy()


def base_inputs(lens, H, seed, s0_std=0.05):
    w = W.PrefillWorkload("edge", None, len(lens), H, 128, 128, "bf16", seed, len_range=(1, 1),
                          s0_std=s0_std)
    return W.prefill_inputs(w, lens=lens)


def run(inp, scale=1.0, interval=0):
    """GPU prefill (tensor-core path) and oracle on the same inputs."""
    import oracle
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], scale=scale,
                    initial_state=d["S0"], snapshot_interval=interval,
                    host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    sp = cs = None
    if interval:
        sp, cs = oracle.snapshot_positions(inp["lens"], interval)
    ro, rS, rsn = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                                 host(inp["b"]), inp["cu_seqlens"].numpy(), scale=scale,
                                 S0=None if inp["S0"] is None else host(inp["S0"]),
                                 snap_pos=sp, cu_snap=cs)
    snaps = None if p.snapshot_view is None else host(p.snapshot_view)
    return (host(p.o), host(p.final_state), snaps), (ro, rS, rsn)


def const_like(t, value):
    return torch.full_like(t, value)


def test_alpha_one_is_the_plain_delta_rule():
    inp = base_inputs([300, 77], 2, 201)
    inp["g"] = const_like(inp["g"], -60.0)  # alpha = 1 / (1 + e^-60) = 1 in fp32 and fp64
    (o, S, sn), (ro, rS, rsn) = run(inp, interval=64)
    assert rel(o, ro) <= TOL and rel(S, rS) <= TOL and rel(sn, rsn) <= TOL


def test_beta_zero_is_pure_decay():
    lens = [200, 64, 1]
    H = 2
    inp = base_inputs(lens, H, 202, s0_std=0.5)
    inp["b"] = const_like(inp["b"], -100.0)  # beta = sigmoid(-100) = 0 in fp32
    (o, S, _), (ro, rS, _) = run(inp, scale=0.75)
    assert rel(o, ro) <= TOL and rel(S, rS) <= TOL
    # closed form: every channel of the initial state decays by its own alphas
    g = host(inp["g"]).astype(np.float64)
    la = -np.logaddexp(0.0, g)                               # log alpha = -softplus(g)
    S0 = host(inp["S0"]).astype(np.float64)
    q = host(inp["q"]).astype(np.float64)
    qh = q / np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), 1e-6)
    cu = np.concatenate([[0], np.cumsum(lens)])
    for s in range(len(lens)):
        G = np.cumsum(la[cu[s]:cu[s + 1]], axis=0)           # [L, H, dk]
        St = np.exp(G)[..., None] * S0[s][None]              # [L, H, dk, dv]
        o_cf = 0.75 * np.einsum("thc,thcn->thn", qh[cu[s]:cu[s + 1]], St)
        assert rel(o[cu[s]:cu[s + 1]], o_cf) <= TOL
        # the state only meets fp32 decay factors, no bf16 operand: far inside the tolerance
        assert rel(S[s], St[-1]) <= 1e-4


def test_beta_one_with_q_equal_k_reads_back_the_value():
    lens = [250, 65]
    inp = base_inputs(lens, 2, 203)
    inp["b"] = const_like(inp["b"], 100.0)   # beta = 1
    inp["q"] = inp["k"].clone()
    (o, S, _), (ro, rS, _) = run(inp)
    assert rel(o, ro) <= TOL and rel(S, rS) <= TOL
    v = host(inp["v"])
    assert rel(o, v) <= TOL                   # o_t = S_t^T k^_t = v_t
    assert rel(ro, v) <= 1e-12                # (the oracle: exactly, to fp64 rounding)


def test_zero_query_and_key_rows():
    lens = [190]
    inp = base_inputs(lens, 2, 204)
    zq = torch.arange(0, 190, 7)
    zk = torch.arange(3, 190, 11)
    inp["q"][zq] = 0
    inp["k"][zk] = 0
    (o, S, _), (ro, rS, _) = run(inp)
    assert rel(o, ro) <= TOL and rel(S, rS) <= TOL
    assert np.all(o[zq.numpy()] == 0)         # q^ = 0: nothing is read
    assert np.all(ro[zq.numpy()] == 0)


def test_orthonormal_retrieval_at_128_channels():
    """alpha = beta = 1: tokens 0..127 write v_t under keys e_pi(t) (q = k, so
    o_t = v_t); tokens 128..255 write nothing (beta = 0) and query e_pi(j_t),
    reading v_{j_t} back across chunk boundaries; the final state holds v_t in
    row pi(t).  Every value involved is a bf16 number and every product has
    one nonzero term, so the kernels' results are the exact ones."""
    H, T = 2, 256
    gen = torch.Generator().manual_seed(205)
    pi = torch.stack([torch.randperm(128, generator=gen) for _ in range(H)], 1)   # [128, H]
    j = torch.randint(0, 128, (128, H), generator=gen)
    v = torch.randn(T, H, 128, generator=gen).to(torch.bfloat16)
    k = torch.zeros(T, H, 128)
    q = torch.zeros(T, H, 128)
    for h in range(H):
        k[torch.arange(128), h, pi[:, h]] = 1.0
        q[torch.arange(128), h, pi[:, h]] = 1.0
        q[128 + torch.arange(128), h, pi[j[:, h], h]] = 1.0
        k[128 + torch.arange(128), h, torch.randint(0, 128, (128,), generator=gen)] = 1.0
    b = torch.cat([torch.full((128, H), 100.0), torch.full((128, H), -100.0)])
    inp = dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v,
               g=torch.full((T, H, 128), -60.0).to(torch.bfloat16), b=b.to(torch.bfloat16),
               cu_seqlens=torch.tensor([0, T]), S0=None, lens=[T])
    (o, S, _), (ro, rS, _) = run(inp)
    vf = host(v)
    expect_o = np.concatenate([vf[:128], np.stack([vf[j[:, h], h] for h in range(H)], 1)])
    expect_S = np.zeros((1, H, 128, 128))
    for h in range(H):
        expect_S[0, h, pi[:, h].numpy()] = vf[:128, h]
    assert rel(ro, expect_o) <= 1e-12 and rel(rS, expect_S) <= 1e-12
    assert rel(o, expect_o) <= 1e-6
    assert rel(S, expect_S) <= 1e-6


def test_decode_edge_cases(oracle_mod):
    """The 128 x 128 decode ring kernel at the same special cases: beta = 0
    leaves Diag(alpha) S; beta = 1 with q = k reads back v; alpha = 1 and a
    zero query."""
    dw = W.DecodeWorkload("edge", 48, 4, 128, 128, 1, 206, s0_std=0.5)
    inp = W.decode_inputs(dw)
    x = {n: inp[n][0].clone() for n in "qkvgb"}
    x["b"][:16] = -100.0                         # rows 0-15: beta = 0
    x["b"][16:32] = 100.0                        # rows 16-31: beta = 1, q = k
    x["q"][16:32] = x["k"][16:32]
    x["g"][32:] = -60.0                          # rows 32-47: alpha = 1
    x["q"][40:] = 0                              # rows 40-47: zero query
    state = inp["state"].cuda().contiguous()
    ref_state = host(inp["state"]).astype(np.float64)
    o = torch.empty(48, 4, 128, dtype=torch.bfloat16, device="cuda")
    kda.kda_decode_step(*[x[n].cuda().contiguous() for n in "qkvgb"], state, o)
    torch.cuda.synchronize()
    ro = oracle_mod.decode(*[host(x[n]) for n in "qkvgb"], ref_state)
    od, sd = host(o), host(state)
    assert rel(od, ro) <= TOL and rel(sd, ref_state) <= 1e-5
    alpha = 1.0 / (1.0 + np.exp(host(x["g"][:16]).astype(np.float64)))
    S0 = host(inp["state"])[:16].astype(np.float64)
    assert rel(sd[:16], alpha[..., None] * S0) <= 1e-6
    assert rel(od[16:32], host(x["v"][16:32])) <= TOL
    assert np.all(od[40:] == 0)
