"""CUDA path vs the fp64 CPU oracle, element by element, on seeded inputs.

Tolerances (relative Frobenius error, on o, final states and snapshots):
1e-5 where inputs are fp32, 5e-3 where inputs are bf16 (state fp32).  Every
call goes through the C ABI (ctypes binding).
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_delta_gb300 import kda
from linear_attention_serving_delta_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def host(t):
    return None if t is None else t.detach().float().cpu().numpy()


def to_dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def make_inputs(lens, H, dk, dv, dtype, seed, s0_std=0.0, g_shift=0.0):
    w = W.PrefillWorkload("case", None, len(lens), H, dk, dv, dtype, seed, len_range=(1, 1),
                          s0_std=s0_std)
    inp = W.prefill_inputs(w, lens=lens)
    if g_shift:
        inp["g"] = (inp["g"].float() + g_shift).to(inp["g"].dtype)
    return inp


def run_both(inp, dtype, scale=1.0, interval=0, boundaries=None):
    """Returns (gpu (o, S, snaps), oracle (o, S, snaps))."""
    lens = inp["lens"]
    cu = inp["cu_seqlens"]
    bpos = cub = None
    if boundaries is not None:
        bl, cb = [], [0]
        for s, pts in enumerate(boundaries):
            bl += list(pts)
            cb.append(len(bl))
        bpos = torch.tensor(bl, dtype=torch.int64)
        cub = torch.tensor(cb, dtype=torch.int64)
    d = to_dev(inp)
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], scale=scale,
                    initial_state=d["S0"], snapshot_interval=interval,
                    boundary_pos=None if bpos is None else bpos.cuda(),
                    cu_boundaries=None if cub is None else cub.cuda(),
                    host_cu_seqlens=cu, host_boundary_pos=bpos, host_cu_boundaries=cub)
    p.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    import oracle
    sp = cs = None
    if interval > 0 or bpos is not None:
        sp, cs = oracle.snapshot_positions(lens, interval, None if bpos is None else bpos.numpy(),
                                           None if cub is None else cub.numpy())
    ref = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                         host(inp["b"]), cu.numpy(), scale=scale, S0=host(inp["S0"]),
                         snap_pos=sp, cu_snap=cs)
    gpu = (host(p.o), host(p.final_state), host(p.snapshot_view))
    return gpu, ref


def worst_unit(a, b, groups):
    """The largest relative Frobenius error over units of the arrays: each
    unit is a[idx] for idx in ``groups`` (units whose reference is all zero
    and whose result is all zero are skipped).  Returns (error, unit)."""
    worst, at = 0.0, None
    for key, idx in groups:
        x, y = np.asarray(a[idx], np.float64), np.asarray(b[idx], np.float64)
        ny = np.linalg.norm(y)
        if ny == 0 and np.linalg.norm(x) == 0:
            continue
        e = np.linalg.norm(x - y) / (ny if ny > 0 else 1.0)
        if e > worst or at is None:
            worst, at = e, key
    return worst, at


# The largest error of any one (sequence, head) or (snapshot, head), as a
# multiple of the global tolerance.  The global relative Frobenius error is
# the figure the tolerance is stated for.  A single unit averages over fewer
# roundings, and a unit of a few tokens hardly at all.  A one-token sequence
# rounds beta (in T diag(beta)) and its A_qk entry to bf16 once for its whole
# output row, so those roundings act coherently (measured worst: 7.0e-3 and
# 1.02e-2 on one-token sequences).  Hence a unit spanning a full chunk (64
# tokens) or more is allowed twice the global bound, a shorter one (and a
# snapshot, whose position the check does not see) four times.  A unit off
# by a chunk, a wrong sequence or a dropped term is off by far more.
UNIT_FACTOR, UNIT_FACTOR_SHORT = 2.0, 4.0


def assert_close(gpu, ref, tol, what="", lens=None):
    """The global relative Frobenius error of o, the final states and the
    snapshots (bound ``tol``), and -- with the sequence lengths -- the same
    error for every (sequence, head) of o and of the final states and every
    (snapshot, head) (bounds UNIT_FACTOR / UNIT_FACTOR_SHORT x ``tol``): one
    wrong sequence, ragged tail or snapshot cannot hide under the norm of
    the others."""
    o, S, sn = gpu
    ro, rS, rsn = ref
    e_o, e_S = rel(o, ro), rel(S, rS)
    assert e_o <= tol, f"{what} o rel err {e_o:.3e} > {tol}"
    assert e_S <= tol, f"{what} final state rel err {e_S:.3e} > {tol}"
    if rsn is not None and len(rsn):
        e_sn = rel(sn, rsn)
        assert e_sn <= tol, f"{what} snapshots rel err {e_sn:.3e} > {tol}"
    if lens is None:
        return
    H = ro.shape[1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    for long_units in (True, False):
        ut = (UNIT_FACTOR if long_units else UNIT_FACTOR_SHORT) * tol
        seqs = [s for s in range(len(lens)) if (lens[s] >= 64) == long_units]
        units_o = [((s, h), (slice(cu[s], cu[s + 1]), h)) for s in seqs for h in range(H) if lens[s] > 0]
        units_S = [((s, h), (s, h)) for s in seqs for h in range(H)]
        for name, a, b, units in (("o", o, ro, units_o), ("final state", S, rS, units_S)):
            e, at = worst_unit(a, b, units)
            assert e <= ut, f"{what} {name}: worst (sequence, head) {at} rel err {e:.3e} > {ut}"
    if rsn is not None and len(rsn):
        ut = UNIT_FACTOR_SHORT * tol
        e, at = worst_unit(sn, rsn, [((j, h), (j, h)) for j in range(len(rsn)) for h in range(H)])
        assert e <= ut, f"{what} snapshots: worst (snapshot, head) {at} rel err {e:.3e} > {ut}"


# ------------------------------------------------------------------ decode (K4)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 128), (128, 16),
                                   (256, 256), (256, 16), (64, 256), (64, 64), (128, 64), (64, 128)])
def test_decode_small(dtype, dk, dv, oracle_mod):
    dw = W.DecodeWorkload("small", 5, 3, dk, dv, 4, 77 + dk + dv)
    inp = W.decode_inputs(dw, dtype=dtype)
    state = inp["state"].cuda().contiguous()
    ref_state = host(inp["state"]).astype(np.float64)
    slots = torch.tensor([3, 0, -1, 4, 1], dtype=torch.int32)
    for step in range(dw.steps):
        args = [inp[x][step].cuda().contiguous() for x in "qkvgb"]
        o = torch.zeros(5, 3, dv, dtype=args[0].dtype, device="cuda")
        kda.kda_decode_step(*args, state, o, state_slots=slots.cuda(), scale=0.7)
        ro = oracle_mod.decode(*[host(inp[x][step]) for x in "qkvgb"], ref_state,
                               slots=slots.numpy(), scale=0.7)
        torch.cuda.synchronize()
        assert rel(host(o), ro) <= TOL[dtype]
        assert np.all(host(o)[2] == 0)                      # skipped row untouched
    assert rel(host(state), ref_state) <= 1e-5              # fp32 state math
    np.testing.assert_array_equal(host(state)[2], host(inp["state"])[2])  # slot 2 unused


def test_decode_full_size(oracle_mod):
    """256 sequences x 32 heads x 128x128 fp32 states, three consecutive steps."""
    dw = W.DECODE_WORKLOADS["decode_256"]
    inp = W.decode_inputs(dw, steps=3)
    state = inp["state"].cuda()
    ref_state = host(inp["state"]).astype(np.float64)
    for step in range(3):
        args = [inp[x][step].cuda() for x in "qkvgb"]
        o = kda.decode_step(*args, state)
        ro = oracle_mod.decode(*[host(inp[x][step]) for x in "qkvgb"], ref_state)
        torch.cuda.synchronize()
        assert rel(host(o), ro) <= TOL["bf16"]
    assert rel(host(state), ref_state) <= 1e-5


@pytest.mark.parametrize("dk,dv,H,gate_per_head", [(64, 64, 4, False), (64, 64, 8, True), (64, 128, 6, False),
                                                   (128, 64, 2, True), (64, 64, 6, False)])
def test_decode_several_heads_per_item(dk, dv, H, gate_per_head, oracle_mod):
    """Small heads share a ring item (several consecutive heads of a row, up
    to 64 KB of state: 4 of 64 x 64, 2 of 64 x 128 or 128 x 64) when the
    head count divides into such groups (H = 6 at 64 x 64 takes pairs).
    Four steps with slot indirection and a skipped row, against the oracle;
    o per (row, head) too."""
    B = 7
    dw = W.DecodeWorkload("group", B, H, dk, dv, 4, 501 + dk + dv + H)
    inp = W.decode_inputs(dw)
    state = inp["state"].cuda().contiguous()
    ref_state = host(inp["state"]).astype(np.float64)
    slots = torch.tensor([3, 0, -1, 6, 1, 5, 2], dtype=torch.int32)
    units = [((r, h), (r, h)) for r in range(B) for h in range(H) if r != 2]
    for step in range(dw.steps):
        x = {n: inp[n][step].contiguous() for n in "qkvgb"}
        gx = x["g"][:, :, 0].contiguous() if gate_per_head else x["g"]
        gref = gx[:, :, None].expand(x["g"].shape) if gate_per_head else x["g"]
        o = torch.zeros(B, H, dv, dtype=x["q"].dtype, device="cuda")
        kda.kda_decode_step(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), gx.cuda(), x["b"].cuda(), state, o,
                            state_slots=slots.cuda(), scale=0.9)
        ro = oracle_mod.decode(host(x["q"]), host(x["k"]), host(x["v"]), host(gref), host(x["b"]), ref_state,
                               slots=slots.numpy(), scale=0.9)
        torch.cuda.synchronize()
        assert rel(host(o), ro) <= TOL["bf16"]
        e, at = worst_unit(host(o), ro, units)
        assert e <= UNIT_FACTOR * TOL["bf16"], f"step {step}: worst (row, head) {at} {e:.3e}"
        assert np.all(host(o)[2] == 0)
    assert rel(host(state), ref_state) <= 1e-5
    np.testing.assert_array_equal(host(state)[4], host(inp["state"])[4])  # slot 4 unused


@pytest.mark.slow
def test_decode_full_size_1000_steps(oracle_mod):
    """The batched decode workload as the benchmark runs it: 256 sequences x 32
    heads x 128 x 128 fp32 states, 1000 consecutive steps of distinct inputs
    (drawn on the device, as the benchmark draws them), the state updated in
    place.  Every step's o is compared with the oracle's (fp64 state carried
    through all 1000 steps), globally and for every (row, head); the state
    after the last step likewise, where the fp32 state must stay within 1e-5
    of the fp64 one after 1000 roundings."""
    dw = W.DECODE_WORKLOADS["decode_256"]
    n = dw.steps
    assert n == 1000
    inp = W.decode_inputs(dw, steps=n, device="cuda", gen_device="cuda")
    state = inp["state"].clone()
    ref_state = host(inp["state"]).astype(np.float64)
    o = torch.empty(dw.batch, dw.H, dw.dv, dtype=torch.bfloat16, device="cuda")
    units = [((r, h), (r, h)) for r in range(dw.batch) for h in range(dw.H)]
    worst_o = 0.0
    for step in range(n):
        args = [inp[x][step] for x in "qkvgb"]
        kda.kda_decode_step(*args, state, o)
        ro = oracle_mod.decode(*[host(a) for a in args], ref_state)
        od = host(o)
        e = rel(od, ro)
        assert e <= TOL["bf16"], f"step {step}: o rel err {e:.3e}"
        if step % 50 == 0 or step == n - 1:
            eu, at = worst_unit(od, ro, units)
            assert eu <= TOL["bf16"], f"step {step}: worst (row, head) {at} o rel err {eu:.3e}"
            worst_o = max(worst_o, eu)
    sd = host(state)
    assert rel(sd, ref_state) <= 1e-5
    eu, at = worst_unit(sd, ref_state, units)
    assert eu <= 1e-5, f"state after {n} steps: worst (row, head) {at} rel err {eu:.3e}"
    print(f"decode_256 x {n} steps: worst (row, head) o {worst_o:.3e}, state {eu:.3e}")


# ------------------------------------------------------------------ prep (K1)
@pytest.mark.parametrize("dtype,dk", [("f32", 64), ("bf16", 64), ("bf16", 128), ("f32", 256),
                                      ("bf16", 256)])
def test_prep(dtype, dk, oracle_mod):
    """bf16 with dk = 128 takes the vectorised kernel: its 64-token tiles
    start mid-chunk and mid-sequence here (lengths 5, 64, 130, ...)."""
    lens = [5, 64, 130, 1, 0, 77, 300]
    inp = make_inputs(lens, 3, dk, 16, dtype, 11)
    d = to_dev(inp)
    qh, kh, G, beta = kda.prep(d["q"], d["k"], d["g"], d["b"], d["cu_seqlens"])
    torch.cuda.synchronize()
    rq, rk, rla, rb = oracle_mod.prep(host(inp["q"]), host(inp["k"]), host(inp["g"]),
                                      host(inp["b"]))
    # G restarts at every 64-token chunk of every sequence (plain definition)
    rG = np.zeros_like(rla)
    cu = inp["cu_seqlens"].numpy()
    for s in range(len(lens)):
        for c0 in range(cu[s], cu[s + 1], 64):
            c1 = min(c0 + 64, cu[s + 1])
            rG[c0:c1] = np.cumsum(rla[c0:c1], axis=0)
    assert rel(host(qh), rq) < 1e-6 and rel(host(kh), rk) < 1e-6
    assert rel(host(beta), rb) < 1e-6
    assert np.max(np.abs(host(G) - rG)) < 1e-5 * max(1.0, np.max(np.abs(rG)))


# ------------------------------------------------------------------ prefill (K0-K3)
def test_prefill_tiny_f32():
    w = W.WORKLOADS["tiny_f32"]
    inp = W.prefill_inputs(w)
    gpu, ref = run_both(inp, "f32")
    assert_close(gpu, ref, TOL["f32"], "tiny_f32", lens=inp["lens"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (16, 128), (256, 256), (256, 64), (32, 256),
                                   (64, 64), (128, 64), (64, 128)])
def test_prefill_ragged_varlen(dtype, dk, dv):
    """Ragged tails and lengths around the chunk size, initial states,
    snapshots every 64 tokens plus interior boundaries, scale != 1."""
    lens = [1, 63, 64, 65, 200, 0, 129]
    inp = make_inputs(lens, 2, dk, dv, dtype, 21, s0_std=0.02)
    bnd = [[1], [10, 63], [], [64, 65], [3, 100, 150, 200], [], [128]]
    gpu, ref = run_both(inp, dtype, scale=0.5, interval=64, boundaries=bnd)
    assert_close(gpu, ref, TOL[dtype], f"{dtype} {dk}x{dv}", lens=lens)


@pytest.mark.parametrize("dtype,d", [("bf16", 64), ("f32", 32)])
def test_prefill_many_sequences(dtype, d):
    """1100 sequences of 0 to 40 tokens (some empty), with initial states and
    snapshots every 64 tokens: the planning kernel's prefix sums over the
    sequences span many warps and two passes of its 1024-thread block."""
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 41, size=1100)]
    lens[5] = lens[1023] = lens[1024] = 0
    lens[1099] = 130
    inp = make_inputs(lens, 2, d, d, dtype, 31, s0_std=0.02)
    gpu, ref = run_both(inp, dtype, interval=64)
    assert_close(gpu, ref, TOL[dtype], f"{dtype} many sequences", lens=lens)


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("dk,dv,H", [(128, 128, 4), (64, 64, 8), (128, 64, 8)])
def test_prefill_64_column_ctas(dk, dv, H):
    """When the inter-chunk kernel's 32-column CTAs would not all fit the GPU
    at once, it runs 64 state columns per CTA (half the CTAs, each at a
    longer step).  Ten ragged sequences with enough heads to exceed the SM
    count: initial states, snapshots every 64 tokens, interior boundaries,
    scale != 1, against the oracle."""
    lens = [1, 63, 64, 65, 200, 0, 129, 3, 77, 300]
    assert len(lens) * H * (dv // 32) > sm_count()  # the 64-column CTAs run
    inp = make_inputs(lens, H, dk, dv, "bf16", 27, s0_std=0.02)
    bnd = [[1], [10, 63], [], [64, 65], [3, 100, 150, 200], [], [128], [2], [], [299]]
    gpu, ref = run_both(inp, "bf16", scale=0.5, interval=64, boundaries=bnd)
    assert_close(gpu, ref, TOL["bf16"], f"64-column CTAs {dk}x{dv}", lens=lens)


def test_prefill_strong_decay():
    """g ~ N(0, 1): about 0.7 of log-decay per token, ~45 over a chunk."""
    inp = make_inputs([300, 64], 2, 128, 128, "bf16", 31, g_shift=3.0)
    gpu, ref = run_both(inp, "bf16")
    assert_close(gpu, ref, TOL["bf16"], "strong decay", lens=inp["lens"])


def test_prefill_decay_past_e_minus_80_per_chunk():
    """g ~ N(+2, 1): about 2.2 nats of log-decay per token, ~140 over a
    64-token chunk and up to ~165 in the strongest channel -- past the e^-87
    where a factor referred to the chunk start leaves the fp32/bf16 range
    ("From KV Cache to Depth Attention", Technical Details: each channel
    keeps its own timescale, fast-forgetting ones included).  The
    tensor-core path refers its factors to half the chunk's decay in each
    channel and matches the oracle, with a clean status word."""
    inp = make_inputs([300, 64, 130], 2, 128, 128, "bf16", 32, s0_std=0.02, g_shift=5.0)
    gpu, ref = run_both(inp, "bf16", interval=64)
    assert np.all(np.isfinite(gpu[0])) and np.all(np.isfinite(gpu[1]))
    assert_close(gpu, ref, TOL["bf16"], "g ~ N(2, 1)", lens=inp["lens"])


def test_prefill_decay_out_of_range_is_flagged():
    """g ~ N(+6, 1): ~390 nats (~560 in log2) of decay over a chunk, past the
    2^-250 the tensor-core operands can span: the call raises status flag
    16 instead of returning such results silently."""
    inp = make_inputs([200], 2, 128, 128, "bf16", 33, g_shift=9.0)
    d = to_dev(inp)
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"],
                    host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert p.device_status() & 16
    # the same inputs in fp32 take the CUDA-core path, which has no such limit
    f = {x: d[x].float() for x in "qkvgb"}
    pf = kda.Prefill(f["q"], f["k"], f["v"], f["g"], f["b"], d["cu_seqlens"],
                     host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert pf.device_status() == 0
    ro, rS, _ = oracle_prefill_of(inp)
    assert rel(host(pf.o), ro) <= 1e-5 and rel(host(pf.final_state), rS) <= 1e-5


def test_prefill_8k_full():
    """Single-sequence prefill, H=32, T=8192, dk=dv=128, bf16 in, fp32 state."""
    inp = W.prefill_inputs(W.WORKLOADS["prefill_8k"])
    gpu, ref = run_both(inp, "bf16")
    assert_close(gpu, ref, TOL["bf16"], "prefill_8k", lens=inp["lens"])


@pytest.mark.slow
def test_prefill_varlen_full():
    """8 packed sequences of U[1024, 32768] tokens, seeded initial states,
    snapshots every 4096 tokens and at the boundaries (one interior + end)."""
    w = W.WORKLOADS["varlen_8"]
    inp = W.prefill_inputs(w)
    bp, cb = inp["boundary_pos"], inp["cu_boundaries"]
    bnd = [bp[cb[s]:cb[s + 1]].tolist() for s in range(len(inp["lens"]))]
    gpu, ref = run_both(inp, "bf16", interval=4096, boundaries=bnd)
    assert_close(gpu, ref, TOL["bf16"], "varlen_8", lens=inp["lens"])


@pytest.mark.slow
def test_prefill_1m_sampled(oracle_mod):
    """The million-token prefill (B=1, H=32, T=2^20, dk=dv=128, bf16, snapshots
    every 65536 tokens) at full size on the device; o, the 16 snapshots and
    the final state of four of the 32 heads are checked against the oracle
    (the oracle's cost is what bounds the sample)."""
    w = W.WORKLOADS["prefill_1m"]
    inp = W.prefill_inputs(w, device="cuda", gen_device="cuda")
    cu = inp["cu_seqlens"].cpu()
    p = kda.Prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["b"], inp["cu_seqlens"],
                    snapshot_interval=w.snapshot_interval, host_cu_seqlens=cu)
    p.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    heads = slice(8, 12)
    sample = {x: host(inp[x][:, heads]) for x in "qkvgb"}
    T = int(cu[-1])
    sp, cs = oracle_mod.snapshot_positions([T], w.snapshot_interval)
    assert len(sp) == 16
    ref = oracle_mod.prefill(sample["q"], sample["k"], sample["v"], sample["g"], sample["b"],
                             cu.numpy(), snap_pos=sp, cu_snap=cs)
    gpu = (host(p.o[:, heads]), host(p.final_state[:, heads]), host(p.snapshot_view[:, heads]))
    del inp, p
    torch.cuda.empty_cache()
    assert_close(gpu, ref, TOL["bf16"], "prefill_1m heads 8-11", lens=[T])


def test_prefill_host_segments_match_one_call():
    """The host-buffer prefill cut into chunk-aligned segments (copies of one
    segment overlapping the prefill of the one before, the fp32 state carried
    between them) gives bit-identical o and final state to a single call."""
    inp = make_inputs([3000], 4, 128, 128, "bf16", 51, s0_std=0.02)
    host_in = {x: inp[x].pin_memory() for x in "qkvgb"}
    args = [host_in[x] for x in "qkvgb"] + [inp["cu_seqlens"]]
    o1, s1 = kda.prefill_host(*args, initial_state=inp["S0"], segments=1)
    o4, s4 = kda.prefill_host(*args, initial_state=inp["S0"], segments=4)
    assert torch.equal(o1, o4)
    assert torch.equal(s1, s4)
    ro, rS, _ = oracle_prefill_of(inp)
    assert rel(o4.float().numpy(), ro) <= TOL["bf16"]
    assert rel(s4.numpy(), rS) <= TOL["bf16"]


def device_prefill_of(inp, scale=1.0):
    d = to_dev(inp)
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], scale=scale,
                    initial_state=d["S0"], host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    return p.o.cpu(), p.final_state.cpu()


@pytest.mark.parametrize("dtype,dk,dv,segments", [("bf16", 128, 128, 3), ("bf16", 128, 128, 0),
                                                  ("f32", 64, 32, 2)])
def test_prefill_host_batch_matches_device_call(dtype, dk, dv, segments):
    """kda_prefill_host over a batch of sequences (pieces of whole sequences,
    an empty sequence among them) gives the same bits as kda_prefill on
    device copies, and the oracle's values."""
    lens = [700, 0, 1500, 64, 2100, 33]
    inp = make_inputs(lens, 3, dk, dv, dtype, 57, s0_std=0.05)
    host_in = {x: inp[x].pin_memory() for x in "qkvgb"}
    o, S = kda.prefill_host(*(host_in[x] for x in "qkvgb"), inp["cu_seqlens"], scale=0.7,
                            initial_state=inp["S0"], segments=segments)
    od, Sd = device_prefill_of(inp, scale=0.7)
    assert torch.equal(o, od)
    assert torch.equal(S, Sd)
    np.testing.assert_array_equal(S[1].numpy(), host(inp["S0"])[1])
    import oracle
    ro, rS, _ = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                               host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]),
                               scale=0.7)
    assert rel(o.float().numpy(), ro) <= TOL[dtype]
    assert rel(S.numpy(), rS) <= TOL[dtype]


def test_prefill_host_pageable_and_empty():
    """Pageable (not pinned) host buffers give the same result as pinned ones;
    an empty prompt returns its initial state."""
    inp = make_inputs([1000], 2, 128, 128, "bf16", 58, s0_std=0.05)
    args = [inp[x] for x in "qkvgb"] + [inp["cu_seqlens"]]
    o_pg, S_pg = kda.prefill_host(*args, initial_state=inp["S0"], segments=5)
    pinned = [inp[x].pin_memory() for x in "qkvgb"] + [inp["cu_seqlens"]]
    o_pn, S_pn = kda.prefill_host(*pinned, initial_state=inp["S0"], segments=5)
    assert torch.equal(o_pg, o_pn) and torch.equal(S_pg, S_pn)
    e = make_inputs([0], 2, 128, 128, "bf16", 59, s0_std=0.3)
    o0, S0 = kda.prefill_host(*(e[x] for x in "qkvgb"), e["cu_seqlens"], initial_state=e["S0"])
    assert o0.shape[0] == 0
    assert torch.equal(S0, e["S0"])


@pytest.mark.parametrize("H,T,P", [(2, 20000, 0), (3, 5000, 5), (1, 300, 8), (2, 4113, 3), (3, 9000, 8)])
def test_prefill_segment_scan(H, T, P):
    """The segment scan (the chain cut into P chunk-aligned segments; their
    state offsets and transition maps in parallel, a serial combine, a second
    pass from the true segment states) gives the oracle's o and final state.
    P = 0 is the automatic choice (9 segments for 2 heads and 313 chunks);
    P = 8 over 5 chunks leaves three segments empty; P = 8 with 3 heads runs
    the first pass (offsets and transition maps, 8 x 3 x 8 = 192 CTAs of 32
    columns) on 64-column CTAs."""
    inp = make_inputs([T], H, 128, 128, "bf16", 61 + H, s0_std=0.05)
    d = to_dev(inp)
    kw = dict(scale=0.9, initial_state=d["S0"], host_cu_seqlens=inp["cu_seqlens"])
    args = [d[x] for x in "qkvgb"] + [d["cu_seqlens"]]
    p = kda.Prefill(*args, scan_segments=P, **kw)
    plain = kda.Prefill(*args, scan_segments=1, **kw)
    assert p.workspace.numel() > plain.workspace.numel()  # the scan's buffers: it is on
    p.run()
    plain.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    import oracle
    ro, rS, _ = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                               host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]),
                               scale=0.9)
    assert rel(host(p.o), ro) <= TOL["bf16"]
    assert rel(host(p.final_state), rS) <= TOL["bf16"]
    # and the unsplit chain agrees to rounding of the fp32 state
    assert rel(host(p.final_state), host(plain.final_state)) < 1e-4
    assert rel(host(p.o), host(plain.o)) < 2e-3


def test_prefill_segment_scan_bad_seqlens():
    """A malformed cu_seqlens on the segment-scan path raises status flag 1
    and leaves the sequence's state as it was, like the plain path."""
    inp = make_inputs([4096], 2, 128, 128, "bf16", 66, s0_std=0.05)
    d = to_dev(inp)
    bad = torch.tensor([0, 4096 + 5], dtype=torch.int64, device="cuda")
    p = kda.Prefill(*(d[x] for x in "qkvgb"), bad, initial_state=d["S0"], scan_segments=4,
                    host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert p.device_status() & 1
    np.testing.assert_array_equal(host(p.final_state), host(inp["S0"]))


def oracle_prefill_of(inp):
    import oracle
    return oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                          host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]))


def test_prefill_empty_sequences_keep_initial_state():
    inp = make_inputs([0, 5, 0], 2, 32, 32, "f32", 41, s0_std=0.5)
    gpu, ref = run_both(inp, "f32")
    np.testing.assert_array_equal(gpu[1][0], host(inp["S0"])[0])
    np.testing.assert_array_equal(gpu[1][2], host(inp["S0"])[2])
    assert_close(gpu, ref, TOL["f32"], lens=inp["lens"])


def test_resume_from_snapshot_gpu(oracle_mod):
    """Prefill to a snapshot, resume from it: matches the uninterrupted oracle
    run (the bf16 tolerance applies to each GPU run against the oracle)."""
    lens = [300]
    inp = make_inputs(lens, 4, 128, 128, "bf16", 51)
    d = to_dev(inp)
    full = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"],
                       boundary_pos=torch.tensor([100], device="cuda"),
                       cu_boundaries=torch.tensor([0, 1], device="cuda"),
                       host_cu_seqlens=inp["cu_seqlens"],
                       host_boundary_pos=torch.tensor([100]),
                       host_cu_boundaries=torch.tensor([0, 1])).run()
    snap = full.snapshot_view.clone()
    rest = {x: d[x][100:].contiguous() for x in "qkvgb"}
    part = kda.Prefill(rest["q"], rest["k"], rest["v"], rest["g"], rest["b"],
                       torch.tensor([0, 200], device="cuda"), initial_state=snap).run()
    torch.cuda.synchronize()
    ro, rS, rsn = oracle_mod.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]),
                                     host(inp["g"]), host(inp["b"]), [0, 300],
                                     snap_pos=[100], cu_snap=[0, 1])
    assert rel(host(snap), rsn) <= TOL["bf16"]
    assert rel(host(part.o), ro[100:]) <= TOL["bf16"]
    assert rel(host(part.final_state), rS) <= TOL["bf16"]
    assert rel(host(part.o), host(full.o)[100:]) <= 2 * TOL["bf16"]


def test_prefill_then_decode_equals_longer_prefill():
    lens = [150]
    inp = make_inputs(lens, 2, 128, 128, "f32", 61)
    d = to_dev(inp)
    n_dec = 5
    head = {x: d[x][: 150 - n_dec].contiguous() for x in "qkvgb"}
    p = kda.Prefill(head["q"], head["k"], head["v"], head["g"], head["b"],
                    torch.tensor([0, 150 - n_dec], device="cuda")).run()
    state = p.final_state.clone()
    outs = []
    for t in range(150 - n_dec, 150):
        args = [d[x][t:t + 1].contiguous() for x in "qkvgb"]
        outs.append(kda.decode_step(*args, state))
    full = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert rel(host(torch.cat(outs)), host(full.o)[150 - n_dec:]) < 1e-5
    assert rel(host(state), host(full.final_state)) < 1e-5


def test_malformed_device_data_is_flagged():
    """Decreasing cu_seqlens: the sequence is skipped and the status word says so."""
    inp = make_inputs([10, 10], 1, 16, 16, "f32", 71)
    d = to_dev(inp)
    bad_cu = torch.tensor([0, 15, 12], dtype=torch.int64, device="cuda")
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], bad_cu).run()
    assert p.device_status() & 1


def test_bounded_waits_give_up_cleanly():
    """A wait limit of 1 ns makes the tensor-core kernels' bounded waits on
    their copies and MMAs give up: the call still returns, the workspace
    status carries flag 8, and the context stays usable -- the next call with
    the default limit gives the oracle's results.  No wait is left to hang
    and nothing faults (the copies and MMAs in flight are drained with the
    long limit before shared memory and TMEM are given back)."""
    inp = make_inputs([4096, 1000], 4, 128, 128, "bf16", 91, s0_std=0.02)
    d = to_dev(inp)
    args = [d[x] for x in "qkvgb"] + [d["cu_seqlens"]]
    hurried = kda.Prefill(*args, initial_state=d["S0"], host_cu_seqlens=inp["cu_seqlens"],
                          wait_limit_ns=1).run()
    torch.cuda.synchronize()
    assert hurried.device_status() & 8
    calm = kda.Prefill(*args, initial_state=d["S0"], host_cu_seqlens=inp["cu_seqlens"]).run()
    torch.cuda.synchronize()
    assert calm.device_status() == 0
    ro, rS, _ = oracle_prefill_of(inp)
    assert rel(host(calm.o), ro) <= TOL["bf16"]
    assert rel(host(calm.final_state), rS) <= TOL["bf16"]


def test_decode_bounded_waits_give_up_cleanly(oracle_mod):
    """The 128 x 128 decode kernel with a 1 ns wait limit: its waits on the
    slot copies give up, the status word gets flag 8, nothing hangs or
    faults, and a later step on the same context with the default limit
    matches the oracle."""
    dw = W.DecodeWorkload("waits", 64, 8, 128, 128, 1, 93)
    inp = W.decode_inputs(dw)
    args = [inp[x][0].cuda().contiguous() for x in "qkvgb"]
    o = torch.zeros(64, 8, 128, dtype=args[0].dtype, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hurried = inp["state"].cuda().contiguous()
    kda.kda_decode_step(*args, hurried, o, wait_limit_ns=1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 8
    status.zero_()
    state = inp["state"].cuda().contiguous()
    kda.kda_decode_step(*args, state, o, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_state = host(inp["state"]).astype(np.float64)
    ro = oracle_mod.decode(*[host(inp[x][0]) for x in "qkvgb"], ref_state)
    assert rel(host(o), ro) <= TOL["bf16"]
    assert rel(host(state), ref_state) <= 1e-5


# ------------------------------------------------------------------ gate per head
def head_gate(inp):
    """g [T, H] (one decay logit per token and head) and the same values
    broadcast to [T, H, dk] for the oracle and the per-channel kernels."""
    gh = inp["g"][:, :, 0].contiguous()
    return gh, gh[:, :, None].expand(inp["g"].shape).contiguous()


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 32), ("bf16", 64, 64)])
def test_prefill_gate_per_head(dtype, dk, dv):
    """g given per (token, head) -- the gated delta rule -- equals the oracle
    with that value in every channel, and the per-channel kernels on the
    broadcast g bit for bit (initial states, snapshots, ragged lengths)."""
    lens = [1, 63, 64, 65, 200, 0, 1300]
    inp = make_inputs(lens, 3, dk, dv, dtype, 95, s0_std=0.02)
    gh, gb = head_gate(inp)
    d = to_dev(inp)
    kw = dict(initial_state=d["S0"], snapshot_interval=64, scale=0.8,
              host_cu_seqlens=inp["cu_seqlens"])
    args = [d["q"], d["k"], d["v"]]
    ph = kda.Prefill(*args, gh.cuda(), d["b"], d["cu_seqlens"], **kw).run()
    pc = kda.Prefill(*args, gb.cuda(), d["b"], d["cu_seqlens"], **kw).run()
    torch.cuda.synchronize()
    assert ph.device_status() == 0
    assert torch.equal(ph.o, pc.o) and torch.equal(ph.final_state, pc.final_state)
    assert torch.equal(ph.snapshot_view, pc.snapshot_view)
    import oracle
    sp, cs = oracle.snapshot_positions(lens, 64)
    ro, rS, rsn = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(gb),
                                 host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]),
                                 scale=0.8, snap_pos=sp, cu_snap=cs)
    assert rel(host(ph.o), ro) <= TOL[dtype]
    assert rel(host(ph.final_state), rS) <= TOL[dtype]
    assert rel(host(ph.snapshot_view), rsn) <= TOL[dtype]


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32), (256, 256), (64, 256)])
def test_decode_and_prep_gate_per_head(dk, dv, oracle_mod):
    """Decode (the ring kernel -- one item per head at 128 x 128, column
    slices moved by tensor-map copies at 256 x 256 and 64 x 256 -- and the
    generic one at 64 x 32) and the prep step with g [rows, H] against the
    oracle on the broadcast g."""
    dw = W.DecodeWorkload("gate", 40, 4, dk, dv, 1, 96 + dk)
    inp = W.decode_inputs(dw)
    gh = inp["g"][0][:, :, 0].contiguous()
    gb = gh[:, :, None].expand(inp["g"][0].shape).contiguous()
    args = [inp[x][0].cuda().contiguous() for x in "qkv"]
    state = inp["state"].cuda().contiguous()
    o = torch.zeros(40, 4, dv, dtype=args[0].dtype, device="cuda")
    kda.kda_decode_step(args[0], args[1], args[2], gh.cuda(), inp["b"][0].cuda().contiguous(), state, o)
    torch.cuda.synchronize()
    ref_state = host(inp["state"]).astype(np.float64)
    ro = oracle_mod.decode(host(inp["q"][0]), host(inp["k"][0]), host(inp["v"][0]), host(gb),
                           host(inp["b"][0]), ref_state)
    assert rel(host(o), ro) <= TOL["bf16"]
    assert rel(host(state), ref_state) <= 1e-5
    # prep: G equal across channels, q^, k^, beta unchanged
    pin = make_inputs([70, 130], 3, dk, 16, "bf16", 97)
    ghp, gbp = head_gate(pin)
    d = to_dev(pin)
    qh, kh, G, beta = kda.prep(d["q"], d["k"], ghp.cuda(), d["b"], d["cu_seqlens"])
    qh2, kh2, G2, beta2 = kda.prep(d["q"], d["k"], gbp.cuda(), d["b"], d["cu_seqlens"])
    torch.cuda.synchronize()
    # (for dk = 128 the per-channel g takes the vectorised kernel: another
    # summation order, hence a tolerance instead of equality)
    for x, y in ((qh, qh2), (kh, kh2), (beta, beta2), (G, G2)):
        assert rel(host(x), host(y)) < 1e-6


def test_prefill_host_gate_per_head():
    """The host-buffer entry with g [T, H] equals the device call."""
    inp = make_inputs([2000], 2, 128, 128, "bf16", 98, s0_std=0.02)
    gh, _ = head_gate(inp)
    host_in = {x: inp[x].pin_memory() for x in "qkvb"}
    o, S = kda.prefill_host(host_in["q"], host_in["k"], host_in["v"], gh.pin_memory(), host_in["b"],
                            inp["cu_seqlens"], initial_state=inp["S0"], segments=3)
    d = to_dev(inp)
    p = kda.Prefill(d["q"], d["k"], d["v"], gh.cuda(), d["b"], d["cu_seqlens"], initial_state=d["S0"],
                    host_cu_seqlens=inp["cu_seqlens"], scan_segments=1).run()
    torch.cuda.synchronize()
    assert rel(o.float().numpy(), host(p.o)) < 2e-3
    assert rel(S.numpy(), host(p.final_state)) < 1e-4
