"""The fused tensor-core prefill (schedule = KDA_SCHEDULE_FUSED: the
intra-chunk pipelines and the inter-chunk chains in one kernel, the records
handed over through L2) against the separate kernels and the oracle.

The fused kernel runs the same arithmetic on the same records as the
separate kernels, in the same order per value: its results are compared bit
for bit (o, final states, snapshots, windows) over the shapes it applies
to -- the 8192-token, 32-head prefill; varlen sequences of 1 to 4096 tokens
with initial states, snapshots and interior boundaries; zero-padded heads of
64 channels; dv = 32; a gate per head; the layer steps -- and once against
the fp64 oracle directly (5e-3 relative Frobenius error, bf16 inputs).
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


def inputs(lens, H, dk, dv, seed, s0=0.02, head_gate=False):
    w = W.PrefillWorkload("fused", None, len(lens), H, dk, dv, "bf16", seed, len_range=(1, 1), s0_std=s0)
    inp = W.prefill_inputs(w, lens=lens)
    if head_gate:
        inp["g"] = inp["g"][:, :, 0].contiguous()
    return inp


def run(inp, schedule, interval=0, bpos=None, cub=None, layer=None):
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    kw = {}
    if layer is not None:
        kw = dict(conv_weights=tuple(t.cuda() for t in layer["taps"]), conv_silu=True,
                  conv_window=tuple(t.cuda() for t in layer["windows"]), conv_window_out=True,
                  out_gate=layer["gate"].cuda())
    p = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], initial_state=d["S0"],
                    snapshot_interval=interval, boundary_pos=None if bpos is None else bpos.cuda(),
                    cu_boundaries=None if cub is None else cub.cuda(),
                    host_cu_seqlens=inp["cu_seqlens"], host_boundary_pos=bpos, host_cu_boundaries=cub,
                    schedule=schedule, **kw)
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


def assert_fused_equals_separate(inp, **kw):
    sep, path_s = run(inp, kda.SCHEDULE_SEPARATE, **kw)
    fus, path_f = run(inp, kda.SCHEDULE_FUSED, **kw)
    assert path_s == kda.PATH_SEPARATE and path_f == kda.PATH_FUSED
    for a, b in zip(outputs(sep), outputs(fus)):
        assert torch.equal(a, b)
    return fus


def test_fused_headline_shape_bit_for_bit():
    assert_fused_equals_separate(inputs([8192], 32, 128, 128, 401, s0=0.0))


def test_fused_varlen_snapshots_boundaries_bit_for_bit():
    lens = [1, 63, 64, 65, 1000, 4096]
    bpos = torch.tensor([1, 2, 40, 64, 65, 500, 999, 1000, 4095], dtype=torch.int64)
    cub = torch.tensor([0, 1, 2, 4, 5, 8, 9], dtype=torch.int64)
    assert_fused_equals_separate(inputs(lens, 4, 128, 128, 402), interval=128, bpos=bpos, cub=cub)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 32)])
def test_fused_narrow_heads_bit_for_bit(dk, dv):
    assert_fused_equals_separate(inputs([2000, 777], 8, dk, dv, 403))


def test_fused_gate_per_head_bit_for_bit():
    assert_fused_equals_separate(inputs([3000, 5], 6, 128, 128, 404, head_gate=True))


def test_fused_layer_steps_bit_for_bit():
    lens = [700, 3, 1500]
    inp = inputs(lens, 4, 128, 128, 405)
    li = W.layer_inputs(412, len(lens), sum(lens), 4, 128, 128, 4, "bf16")
    assert_fused_equals_separate(inp, layer=li)


def test_fused_against_oracle():
    import oracle
    lens = [513, 64, 1999]
    inp = inputs(lens, 4, 128, 128, 406)
    p, path = run(inp, kda.SCHEDULE_FUSED, interval=256)
    assert path == kda.PATH_FUSED
    sp, cs = oracle.snapshot_positions(lens, 256)
    ro, rS, rsn = oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                                 host(inp["b"]), inp["cu_seqlens"].numpy(), S0=host(inp["S0"]),
                                 snap_pos=sp, cu_snap=cs)
    assert rel(host(p.o), ro) <= TOL
    assert rel(host(p.final_state), rS) <= TOL
    assert rel(host(p.snapshot_view), rsn) <= TOL
