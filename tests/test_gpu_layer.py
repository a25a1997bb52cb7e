"""The layer steps (short convolution on q, k, v; output gate) on the CUDA
paths vs the fp64 oracle (``oracle.layer``), through the C ABI.

Tolerances as for the recurrence alone: relative Frobenius error 5e-3 with
bf16 inputs, 1e-5 with fp32 inputs, on o, final states and snapshots; the
windows after a call are copies of inputs and must match exactly.  Cases
cover sequences shorter than the window, chunks that start one or two
tokens after a sequence start (a boundary at 1 or 2), windows given and
absent and updated in place, SiLU on and off, the gate per channel and per
head, the gate per head of the decay, the segment scan, and the decode
kernels (ring and generic) chained after a prefill.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_delta_gb300 import kda
from linear_attention_serving_delta_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 5e-3}
ODT = {"f32": "float32", "bf16": "bfloat16"}


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def host(t):
    return None if t is None else t.detach().double().cpu().numpy()


def case(lens, H, dk, dv, dtype, seed, width, gate_mode="channel", head_gate=False, s0=0.02):
    w = W.PrefillWorkload("case", None, len(lens), H, dk, dv, dtype, seed, len_range=(1, 1),
                          s0_std=s0)
    inp = W.prefill_inputs(w, lens=lens)
    if head_gate:
        inp["g"] = inp["g"][:, :, 0].contiguous()
    T = sum(lens)
    li = W.layer_inputs(seed + 7, len(lens), T, H, dk, dv, width, dtype,
                        gate_per_head=gate_mode == "head")
    if gate_mode is None:
        li["gate"] = None
    return inp, li


def oracle_prefill(inp, li, use_windows, silu, dtype, interval=0, bpos=None, cub=None):
    from oracle import layer
    import oracle
    g = host(inp["g"])
    if g.ndim == 2:  # one decay per token and head = the same logit in every channel
        g = np.repeat(g[:, :, None], inp["q"].shape[2], axis=2)
    sp = cs = None
    if interval > 0 or bpos is not None:
        sp, cs = oracle.snapshot_positions(inp["lens"], interval,
                                           None if bpos is None else bpos.numpy(),
                                           None if cub is None else cub.numpy())
    return layer.prefill_layer(
        host(inp["q"]), host(inp["k"]), host(inp["v"]), g, host(inp["b"]),
        inp["cu_seqlens"].numpy(), conv_w=tuple(host(t) for t in li["taps"]),
        windows=tuple(host(t) for t in li["windows"]) if use_windows else None,
        use_silu=silu, dtype=ODT[dtype], out_gate=host(li["gate"]),
        S0=host(inp["S0"]), snap_pos=sp, cu_snap=cs)


def gpu_prefill(inp, li, use_windows, silu, interval=0, bpos=None, cub=None, inplace=False,
                scan_segments=0):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    taps = tuple(t.cuda() for t in li["taps"])
    win = tuple(t.cuda() for t in li["windows"]) if use_windows else None
    if inplace:
        win = tuple(t.clone() for t in win)
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"],
                    initial_state=d["S0"], snapshot_interval=interval,
                    boundary_pos=None if bpos is None else bpos.cuda(),
                    cu_boundaries=None if cub is None else cub.cuda(),
                    host_cu_seqlens=inp["cu_seqlens"], host_boundary_pos=bpos,
                    host_cu_boundaries=cub, scan_segments=scan_segments,
                    conv_weights=taps, conv_silu=silu, conv_window=win,
                    conv_window_out=win if inplace else True,
                    out_gate=None if li["gate"] is None else li["gate"].cuda())
    p.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    return p


def boundaries_near_starts(lens):
    """Boundary positions 1 and 2 where a sequence is long enough (chunks
    starting one and two tokens into it), plus its end."""
    bl, cb = [], [0]
    for L in lens:
        pts = sorted({x for x in (1, 2, L) if 1 <= x <= L})
        bl += pts
        cb.append(len(bl))
    return torch.tensor(bl, dtype=torch.int64), torch.tensor(cb, dtype=torch.int64)


def check(p, ref, dtype, what, snaps=True):
    ro, rS, rsn, rwin = ref
    tol = TOL[dtype]
    e = rel(host(p.o), ro)
    assert e <= tol, f"{what}: o rel err {e:.3e}"
    e = rel(host(p.final_state), rS)
    assert e <= tol, f"{what}: final state rel err {e:.3e}"
    if snaps and rsn is not None:
        e = rel(host(p.snapshot_view), rsn)
        assert e <= tol, f"{what}: snapshots rel err {e:.3e}"
    for t in range(3):
        np.testing.assert_array_equal(host(p.conv_window_out[t]), rwin[t], err_msg=f"{what} window {t}")


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 64), ("f32", 32, 16),
                                         ("bf16", 256, 256)])
def test_prefill_conv_gate_varlen(dtype, dk, dv):
    lens = [1, 2, 3, 61, 130, 200]
    inp, li = case(lens, 4, dk, dv, dtype, seed=300, width=4)
    bpos, cub = boundaries_near_starts(lens)
    p = gpu_prefill(inp, li, True, True, interval=64, bpos=bpos, cub=cub)
    ref = oracle_prefill(inp, li, True, True, dtype, interval=64, bpos=bpos, cub=cub)
    check(p, ref, dtype, f"{dtype} d={dk}")


@pytest.mark.parametrize("width,silu,windows,gate_mode,head_gate", [
    (2, False, False, "channel", False),
    (3, True, True, "head", False),
    (4, False, True, None, True),
    (4, True, False, "head", True),
    (1, True, False, "channel", False),
])
def test_prefill_conv_variants_tc(width, silu, windows, gate_mode, head_gate):
    lens = [5, 70, 129, 64]
    inp, li = case(lens, 3, 128, 128, "bf16", seed=310 + width, width=width, gate_mode=gate_mode,
                   head_gate=head_gate)
    p = gpu_prefill(inp, li, windows, silu)
    ref = oracle_prefill(inp, li, windows, silu, "bf16")
    check(p, ref, "bf16", f"W={width} silu={silu} win={windows} gate={gate_mode} hg={head_gate}")


@pytest.mark.parametrize("gate_mode", ["channel", "head"])
def test_layer_steps_on_64_column_ctas(gate_mode):
    """The convolution and the output gate with enough sequences and heads
    that the inter-chunk kernel runs 64 state columns per CTA (its 32-column
    CTAs would exceed the SM count): the gate's factors are applied by the
    output rows of a 64-column CTA."""
    lens = [5, 70, 129, 64, 1, 2, 200, 33, 90, 3]
    H = 4
    assert len(lens) * H * 4 > torch.cuda.get_device_properties(0).multi_processor_count
    inp, li = case(lens, H, 128, 128, "bf16", seed=330, width=3, gate_mode=gate_mode)
    p = gpu_prefill(inp, li, True, True)
    ref = oracle_prefill(inp, li, True, True, "bf16")
    check(p, ref, "bf16", f"64-column CTAs gate={gate_mode}")


def test_output_gate_on_padded_heads():
    """bf16 heads of 64 channels run on the tensor-core kernels zero-padded
    to 128; the output gate (per channel and per head) rides on their store
    with the caller's 64-column layout."""
    lens = [70, 3, 129]
    for mode in ("channel", "head"):
        inp, li = case(lens, 2, 64, 64, "bf16", seed=325, width=1, gate_mode=mode)
        li["taps"] = None
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"],
                        initial_state=d["S0"], snapshot_interval=64,
                        host_cu_seqlens=inp["cu_seqlens"], out_gate=li["gate"].cuda()).run()
        torch.cuda.synchronize()
        from oracle import layer
        import oracle
        sp, cs = oracle.snapshot_positions(lens, 64)
        ro, rS, rsn, _ = layer.prefill_layer(
            host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]), host(inp["b"]),
            inp["cu_seqlens"].numpy(), out_gate=host(li["gate"]), S0=host(inp["S0"]),
            snap_pos=sp, cu_snap=cs)
        assert rel(host(p.o), ro) <= TOL["bf16"], mode
        assert rel(host(p.final_state), rS) <= TOL["bf16"], mode
        assert rel(host(p.snapshot_view), rsn) <= TOL["bf16"], mode


@pytest.mark.parametrize("dtype,dk", [("bf16", 128), ("f32", 64)])
def test_prep_with_convolution(dtype, dk):
    """kda_prep with the short convolution: q^ and k^ are the normalised
    convolved inputs (the prefill's first step), G and beta unchanged;
    sequences shorter than the window and an empty one."""
    import oracle
    from oracle import layer
    lens = [5, 2, 64, 0, 130, 1]
    inp, li = case(lens, 3, dk, 16, dtype, seed=380, width=4)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    taps = tuple(t.cuda() for t in li["taps"])
    win = tuple(t.cuda() for t in li["windows"])
    qh, kh, G, beta = kda.prep(d["q"], d["k"], d["g"], d["b"], d["cu_seqlens"],
                               conv_weights=taps, conv_silu=True, conv_window=win[:2])
    torch.cuda.synchronize()
    cu = inp["cu_seqlens"].numpy()
    cq, _ = layer.short_conv(host(inp["q"]), host(li["taps"][0]), cu, host(li["windows"][0]), True,
                             ODT[dtype])
    ck, _ = layer.short_conv(host(inp["k"]), host(li["taps"][1]), cu, host(li["windows"][1]), True,
                             ODT[dtype])
    rq, rk, _, rb = oracle.prep(cq, ck, host(inp["g"]), host(inp["b"]))
    # (a convolved value may round to the other neighbouring bf16 value where the
    # fp32 and fp64 sums straddle a rounding boundary: a few elements in 1e5)
    assert rel(host(qh), rq) < 1e-4 and rel(host(kh), rk) < 1e-4
    assert rel(host(beta), rb) < 1e-6
    qp, kp, Gp, _ = kda.prep(d["q"], d["k"], d["g"], d["b"], d["cu_seqlens"])
    torch.cuda.synchronize()
    # G does not depend on the convolution (without it bf16 at dk = 128 takes
    # the vectorised kernel, whose scan sums in another order: equal to rounding)
    assert rel(host(G), host(Gp)) < 1e-6
    assert rel(host(qh), host(qp)) > 1e-2  # the convolution did change q^


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 32)])
def test_prefill_windows_in_place(dtype, d):
    lens = [2, 90, 1]
    inp, li = case(lens, 2, d, d, dtype, seed=320, width=4)
    p = gpu_prefill(inp, li, True, False, inplace=True)
    ref = oracle_prefill(inp, li, True, False, dtype)
    check(p, ref, dtype, "in place")


def test_unit_tap_and_saturated_gate_are_bitwise_identity():
    """Width 1 with tap 1.0 reproduces the inputs exactly and a gate logit of
    30 has sigmoid 1.0 in fp32, so o, the final state and the snapshots are
    bit-identical to a call without the layer steps (the convolution and
    plain instances of the intra-chunk kernel agree bit for bit)."""
    lens = [100, 37]
    H = 2
    for dtype, d in (("bf16", 128), ("f32", 64)):
        inp, _ = case(lens, H, d, d, dtype, seed=330, width=1)
        dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        taps = tuple(torch.ones(1, H, d, device="cuda") for _ in range(3))
        gate = torch.full((sum(lens), H, d), 30.0, device="cuda").to(inp["q"].dtype)
        args = (dev["q"], dev["k"], dev["v"], dev["g"], dev["b"], dev["cu_seqlens"])
        plain = kda.Prefill(*args, initial_state=dev["S0"], snapshot_interval=64,
                            host_cu_seqlens=inp["cu_seqlens"]).run()
        lay = kda.Prefill(*args, initial_state=dev["S0"], snapshot_interval=64,
                          host_cu_seqlens=inp["cu_seqlens"], conv_weights=taps,
                          out_gate=gate).run()
        torch.cuda.synchronize()
        assert torch.equal(plain.o, lay.o), dtype
        assert torch.equal(plain.final_state, lay.final_state), dtype
        assert torch.equal(plain.snapshot_view, lay.snapshot_view), dtype


def test_prefill_conv_segment_scan():
    """One long sequence with few heads takes the segment scan; the halo of
    each segment's first chunk comes from the segment before."""
    lens = [64 * 48 + 17]
    inp, li = case(lens, 2, 128, 128, "bf16", seed=340, width=4)
    p = gpu_prefill(inp, li, True, True, scan_segments=4)
    ref = oracle_prefill(inp, li, True, True, "bf16")
    check(p, ref, "bf16", "segment scan")
    assert kda.kda_prefill_workspace_size(p.args) > kda.kda_prefill_workspace_size(
        kda.make_prefill_args(*(t.cuda() for t in (inp["q"], inp["k"], inp["v"], inp["g"],
                                                   inp["b"], inp["cu_seqlens"])), p.o,
                              scan_segments=1))


@pytest.mark.parametrize("dtype,d,gate_mode", [("bf16", 128, "channel"), ("bf16", 128, "head"),
                                               ("f32", 128, "channel"), ("f32", 32, "head"),
                                               ("bf16", 64, "channel")])
def test_decode_conv_gate(dtype, d, gate_mode):
    """Three decode steps over a slot pool (rows map to permuted slots, one
    row skipped) with the windows advanced in place; bf16 at d = 128 runs
    the ring kernel, the others the generic one."""
    from oracle import layer
    B, H, Wd, steps = 6, 3, 4, 3
    n_slots = 8
    wl = W.DecodeWorkload("case", B, H, d, d, steps, 350, s0_std=0.02)
    di = W.decode_inputs(wl, dtype=dtype)
    li = W.layer_inputs(351, n_slots, B * steps, H, d, d, Wd, dtype,
                        gate_per_head=gate_mode == "head")
    slots = torch.tensor([5, 0, -1, 7, 2, 3], dtype=torch.int32)
    pool = torch.randn(n_slots, H, d, d, generator=torch.Generator().manual_seed(352)) * 0.02
    ref_state = pool.double().numpy().copy()
    ref_win = [host(t).copy() for t in li["windows"]]
    state = pool.cuda()
    win = tuple(t.cuda() for t in li["windows"])
    taps = tuple(t.cuda() for t in li["taps"])
    gates = li["gate"].reshape(steps, B, *li["gate"].shape[1:])
    for s in range(steps):
        x = {k: di[k][s] for k in ("q", "k", "v", "g", "b")}
        o = torch.zeros(B, H, d, dtype=x["q"].dtype, device="cuda")
        kda.kda_decode_step(*(x[k].cuda() for k in ("q", "k", "v", "g", "b")), state, o,
                            state_slots=slots.cuda(), conv_weights=taps, conv_silu=True,
                            conv_window=win, out_gate=gates[s].cuda())
        ro = layer.decode_layer(*(host(x[k]) for k in ("q", "k", "v", "g", "b")), ref_state,
                                conv_w=tuple(host(t) for t in li["taps"]), windows=ref_win,
                                use_silu=True, dtype=ODT[dtype], out_gate=host(gates[s]),
                                slots=slots.numpy())
        torch.cuda.synchronize()
        live = slots.numpy() >= 0
        e = rel(host(o)[live], ro[live])
        assert e <= TOL[dtype], f"step {s}: o rel err {e:.3e}"
    e = rel(host(state), ref_state)
    assert e <= TOL[dtype], f"state rel err {e:.3e}"
    for t in range(3):
        np.testing.assert_array_equal(host(win[t]), ref_win[t])


def test_prefill_then_decode_with_layer_steps():
    """A GPU prefill of the first p tokens (windows out) followed by GPU
    decode steps over the rest (windows in place) matches the oracle's one
    prefill of the whole sequence, token by token."""
    from oracle import layer
    L, p, H, d, Wd = 75, 70, 2, 128, 4
    inp, li = case([L], H, d, d, "bf16", seed=360, width=Wd)
    ref = oracle_prefill(inp, li, True, True, "bf16")
    head = {k: inp[k][:p] for k in ("q", "k", "v", "g", "b")}
    head.update(S0=inp["S0"], cu_seqlens=torch.tensor([0, p]), lens=[p])
    lhead = dict(taps=li["taps"], windows=li["windows"], gate=li["gate"][:p])
    pre = gpu_prefill(head, lhead, True, True)
    e = rel(host(pre.o), ref[0][:p])
    assert e <= TOL["bf16"], f"prefill o {e:.3e}"
    state = pre.final_state.clone()
    win = tuple(t.clone() for t in pre.conv_window_out)
    taps = tuple(t.cuda() for t in li["taps"])
    outs = []
    for t in range(p, L):
        x = [inp[k][t:t + 1].cuda() for k in ("q", "k", "v", "g", "b")]
        o = kda.decode_step(*x, state, conv_weights=taps, conv_silu=True, conv_window=win,
                            out_gate=li["gate"][t:t + 1].cuda())
        outs.append(host(o)[0])
    torch.cuda.synchronize()
    e = rel(np.stack(outs), ref[0][p:])
    assert e <= TOL["bf16"], f"decode o {e:.3e}"
    e = rel(host(state)[0], ref[1][0])
    assert e <= TOL["bf16"], f"state {e:.3e}"
    for t in range(3):
        np.testing.assert_array_equal(host(win[t])[0], ref[3][t][0])
