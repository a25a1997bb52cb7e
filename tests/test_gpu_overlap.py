"""The overlapped tensor-core prefill (schedule = KDA_SCHEDULE_OVERLAP, and
the automatic choice for one sequence: the intra-chunk kernel on every SM up
to a split, then the inter-chunk chains launched as its programmatic
dependent on the SMs it leaves, reading each record once it is published)
against the separate kernels and the oracle.

The overlapped kernels run the same arithmetic on the same records as the
separate kernels: their results are compared bit for bit (o, final state,
snapshots, windows) over the shapes they apply to -- an 8192-token prefill
of 16 heads (64 chains, the automatic choice); one sequence with an initial
state, snapshots and interior boundaries; ragged lengths (one token, one
chunk, a chunk and a token); zero-padded heads of 64 channels and dv = 32;
a gate per head; the layer steps; a long sequence with few heads (where the
chains reach records still being made) -- and once against the fp64 oracle
directly (5e-3 relative Frobenius error, bf16 inputs).  Two calls in a row on one
workspace give the same bits (the planning kernel clears the flags and
counters of the call before).
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
    return t.detach().double().cpu().numpy()


def inputs(T, H, dk, dv, seed, s0=0.02, head_gate=False):
    w = W.PrefillWorkload("overlap", None, 1, H, dk, dv, "bf16", seed, len_range=(1, 1), s0_std=s0)
    inp = W.prefill_inputs(w, lens=[T])
    if head_gate:
        inp["g"] = inp["g"][:, :, 0].contiguous()
    return inp


def make(inp, schedule, interval=0, bpos=None, layer=None, scan_segments=0):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    kw = {}
    if layer is not None:
        kw = dict(conv_weights=tuple(t.cuda() for t in layer["taps"]), conv_silu=True,
                  conv_window=tuple(t.cuda() for t in layer["windows"]), conv_window_out=True,
                  out_gate=layer["gate"].cuda())
    cub = None if bpos is None else torch.tensor([0, len(bpos)], dtype=torch.int64)
    return kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], initial_state=d["S0"],
                       snapshot_interval=interval, boundary_pos=None if bpos is None else bpos.cuda(),
                       cu_boundaries=None if cub is None else cub.cuda(),
                       host_cu_seqlens=inp["cu_seqlens"], host_boundary_pos=bpos, host_cu_boundaries=cub,
                       scan_segments=scan_segments, schedule=schedule, **kw)


def run(inp, schedule, **kw):
    p = make(inp, schedule, **kw)
    path = kda.kda_prefill_schedule(p.args)
    p.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    return p, path


def outputs(p):
    out = [p.o, p.final_state]
    if p.snapshot_view is not None:
        out.append(p.snapshot_view)
    if p.conv_window_out is not None:
        out += list(p.conv_window_out)
    return out


def assert_overlap_equals_separate(inp, schedule=kda.SCHEDULE_OVERLAP, **kw):
    sep, path_s = run(inp, kda.SCHEDULE_SEPARATE, **kw)
    ovl, path_o = run(inp, schedule, **kw)
    assert path_s == kda.PATH_SEPARATE and path_o == kda.PATH_OVERLAP
    for a, b in zip(outputs(sep), outputs(ovl)):
        assert torch.equal(a, b)
    return ovl


def test_overlap_automatic_choice_bit_for_bit():
    # the automatic choice takes the overlapped kernels here (64 chains)
    assert_overlap_equals_separate(inputs(8192, 16, 128, 128, 501, s0=0.0), schedule=kda.SCHEDULE_AUTO)


def test_overlap_snapshots_boundaries_bit_for_bit():
    bpos = torch.tensor([1, 2, 40, 64, 65, 500, 4095, 7000], dtype=torch.int64)
    assert_overlap_equals_separate(inputs(7001, 16, 128, 128, 502), interval=1024, bpos=bpos)


@pytest.mark.parametrize("T", [1, 64, 65, 8191])
def test_overlap_ragged_lengths_bit_for_bit(T):
    assert_overlap_equals_separate(inputs(T, 16, 128, 128, 503 + T))


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 32)])
def test_overlap_narrow_heads_bit_for_bit(dk, dv):
    assert_overlap_equals_separate(inputs(5000, 32, dk, dv, 504))


def test_overlap_gate_per_head_bit_for_bit():
    assert_overlap_equals_separate(inputs(6000, 16, 128, 128, 505, head_gate=True))


def test_overlap_layer_steps_bit_for_bit():
    T = 3000
    inp = inputs(T, 16, 128, 128, 506)
    li = W.layer_inputs(512, 1, T, 16, 128, 128, 4, "bf16")
    assert_overlap_equals_separate(inp, layer=li)


def test_overlap_long_sequence_few_heads_bit_for_bit():
    # 4 heads (the segment scan off): 16 chains, so 136 SMs stay with the
    # intra-chunk kernel and the split comes early; the chains reach records
    # still being made
    assert_overlap_equals_separate(inputs(65536, 4, 128, 128, 507), scan_segments=1)


def test_overlap_repeated_calls_same_bits():
    inp = inputs(4096, 16, 128, 128, 508)
    p = make(inp, kda.SCHEDULE_OVERLAP)
    assert kda.kda_prefill_schedule(p.args) == kda.PATH_OVERLAP
    p.run()
    torch.cuda.synchronize()
    first = [t.clone() for t in outputs(p)]
    p.run()
    torch.cuda.synchronize()
    assert p.device_status() == 0
    for a, b in zip(first, outputs(p)):
        assert torch.equal(a, b)


def test_overlap_against_oracle():
    import oracle
    T = 3001
    inp = inputs(T, 16, 128, 128, 509)
    p, path = run(inp, kda.SCHEDULE_OVERLAP, interval=256)
    assert path == kda.PATH_OVERLAP
    sp, cs = oracle.snapshot_positions([T], 256)
    ro, rS, rsn = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                                 host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]),
                                 snap_pos=sp, cu_snap=cs)
    assert rel(host(p.o), ro) <= TOL
    assert rel(host(p.final_state), rS) <= TOL
    assert rel(host(p.snapshot_view), rsn) <= TOL
