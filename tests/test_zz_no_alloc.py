"""kda_prefill_noalloc: the prefill entry point that allocates nothing.

Callers that cannot allocate device memory at the point of the call (an
engine that reserved all of HBM for its state pools, a host framework that
owns every allocation, a path where an allocation would synchronise the
device) use this entry point; it runs the prefill on a fixed 64 MiB
workspace inside the library.  This test calls it through the C ABI twice in
a row, on two different inputs, and checks each result against kda_prefill
with a caller-owned workspace: the kernels, the workspace layout and the
inputs are the same, so o, the final states and the snapshots must be the
same bits.  The first case is also checked against the oracle within the
bf16 tolerance of the parity tests (relative Frobenius error 5e-3), and the
status word of each call (read back through
kda_prefill_noalloc_device_status, which allocates nothing either) must be
clean.  It also checks the size limit.

This file is collected last on purpose and runs alone in a fresh process as
well as after the other tests.
"""
import numpy as np
import pytest
import torch

from linear_attention_serving_delta_gb300 import kda
from linear_attention_serving_delta_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = 5e-3


def rel(a, b):
    a = a.detach().double().cpu().numpy()
    b = b.detach().double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def inputs(seed, lens, H=4):
    w = W.PrefillWorkload("noalloc", None, len(lens), H, 128, 128, "bf16", seed, len_range=(1, 1),
                          s0_std=0.02)
    inp = W.prefill_inputs(w, lens=lens)
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}, inp


def test_noalloc_matches_workspace_prefill_twice():
    for seed, lens in ((301, [300, 129]), (302, [77, 64, 200])):
        d, h = inputs(seed, lens)
        bpos = torch.tensor([50] + [lens[1]] + [10] * (len(lens) - 2), dtype=torch.int64)
        cub = torch.arange(len(lens) + 1, dtype=torch.int64)
        ref = kda.Prefill(d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"],
                          initial_state=d["S0"], snapshot_interval=128,
                          boundary_pos=bpos.cuda(), cu_boundaries=cub.cuda(),
                          host_cu_seqlens=h["cu_seqlens"], host_boundary_pos=bpos,
                          host_cu_boundaries=cub).run()
        # same arguments, outputs of its own, no workspace
        o = torch.full_like(ref.o, float("nan"))
        fs = torch.full_like(ref.final_state, float("nan"))
        sn = torch.full_like(ref.snapshots, float("nan"))
        args = kda.make_prefill_args(
            d["q"], d["k"], d["v"], d["g"], d["b"], d["cu_seqlens"], o, initial_state=d["S0"],
            final_state=fs, snapshot_interval=128, boundary_pos=bpos.cuda(),
            cu_boundaries=cub.cuda(), cu_snapshots=ref.cu_snapshots, snapshots=sn)
        assert kda.kda_prefill_workspace_size(args) <= kda.NOALLOC_SCRATCH_BYTES
        kda.kda_prefill_noalloc(args)
        torch.cuda.synchronize()
        assert kda.kda_prefill_noalloc_device_status() == 0
        assert ref.device_status() == 0
        n = ref.n_snap
        assert n > 0
        assert torch.equal(o, ref.o)
        assert torch.equal(fs, ref.final_state)
        assert torch.equal(sn[:n], ref.snapshots[:n])
        if seed == 301:
            import oracle
            sp, cs = oracle.snapshot_positions(lens, 128, bpos.numpy(), cub.numpy())
            f = lambda t: t.float().numpy()
            ro, rS, rsn = oracle.prefill(f(h["q"]), f(h["k"]), f(h["v"]), f(h["g"]), f(h["b"]),
                                         h["cu_seqlens"].numpy(), S0=f(h["S0"]),
                                         snap_pos=sp, cu_snap=cs)
            assert rel(o, torch.from_numpy(ro)) <= TOL
            assert rel(fs, torch.from_numpy(rS)) <= TOL
            assert rel(sn[:n], torch.from_numpy(rsn)) <= TOL


def test_noalloc_rejects_workspace_beyond_its_limit():
    # 8192 tokens x 32 heads needs a few hundred MB of workspace: refused on the host
    T, H = 8192, 32
    z = torch.zeros(T, H, 128, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int64, device="cuda")
    o = torch.empty_like(z)
    args = kda.make_prefill_args(z, z, z, z, b, cu, o)
    assert kda.kda_prefill_workspace_size(args) > kda.NOALLOC_SCRATCH_BYTES
    with pytest.raises(kda.KdaError) as err:
        kda.kda_prefill_noalloc(args)
    assert err.value.status == 3  # KDA_ERR_WORKSPACE
