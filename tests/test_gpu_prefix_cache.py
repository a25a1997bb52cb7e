"""Resuming prompts through the snapshot retention policy on the GPU: states
saved into pool rows chosen by the cache (snapshot_slot_map), a later prompt
sharing a prefix resumed from the longest cached one, checked against the
fp64 oracle over the whole prompt."""
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
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def host(t):
    return t.detach().float().cpu().numpy()


def inputs(T, H, seed, d=128):
    w = W.PrefillWorkload("cache", None, 1, H, d, d, "bf16", seed, len_range=(1, 1))
    return W.prefill_inputs(w, lens=[T])


def oracle_run(inp):
    import oracle
    return oracle.prefill(host(inp["q"]), host(inp["k"]), host(inp["v"]), host(inp["g"]),
                          host(inp["b"]), inp["cu_seqlens"].numpy())


@pytest.mark.parametrize("dh", [128, 64])
def test_slot_map_places_and_skips_snapshots(dh):
    """(64-channel heads run on the tensor-core kernels zero-padded: their
    snapshot rows keep the [64, 64] layout and leave other rows untouched.)"""
    inp = inputs(256, 2, 81, dh)
    d = {x: inp[x].cuda() for x in "qkvgb"}
    cu = inp["cu_seqlens"]
    plain = kda.Prefill(*(d[x] for x in "qkvgb"), cu.cuda(), snapshot_interval=64,
                        host_cu_seqlens=cu).run()
    pool = torch.full((8, 2, dh, dh), 7.0, device="cuda")
    smap = torch.tensor([3, -1, 0, 7], dtype=torch.int32, device="cuda")
    mapped = kda.Prefill(*(d[x] for x in "qkvgb"), cu.cuda(), snapshot_interval=64,
                         host_cu_seqlens=cu, snapshot_pool=pool, snapshot_slot_map=smap).run()
    torch.cuda.synchronize()
    assert mapped.device_status() == 0
    snaps = plain.snapshot_view
    for j, row in enumerate([3, -1, 0, 7]):
        if row >= 0:
            assert torch.equal(pool[row], snaps[j])
    assert bool((pool[1] == 7.0).all()) and bool((pool[2] == 7.0).all())
    # a row past the pool raises status flag 2 and is not written
    bad = kda.Prefill(*(d[x] for x in "qkvgb"), cu.cuda(), snapshot_interval=64,
                      host_cu_seqlens=cu, snapshot_pool=pool,
                      snapshot_slot_map=torch.tensor([0, 1, 2, 8], dtype=torch.int32,
                                                     device="cuda")).run()
    torch.cuda.synchronize()
    assert bad.device_status() & 2


def test_resume_from_longest_cached_prefix():
    H = 2
    cache = kda.PrefixCache(6)
    pool = torch.zeros(6, H, 128, 128, device="cuda")
    rng = np.random.default_rng(5)
    tok_a = rng.integers(0, 30000, 3000).astype(np.int32)
    a = inputs(3000, H, 82)
    da = {x: a[x].cuda() for x in "qkvgb"}
    p, o, S = kda.prefill_cached(cache, pool, tok_a, *(da[x] for x in "qkvgb"), interval=1024)
    torch.cuda.synchronize()
    assert p == 0 and cache.entries() == 3                 # 1024, 2048 and the end
    ro, rS, _ = oracle_run(a)
    assert rel(host(o), ro) <= TOL and rel(host(S), rS) <= TOL

    # prompt B: A's first 2500 tokens, then 1500 of its own
    b = inputs(4000, H, 83)
    for x in "qkvgb":
        b[x][:2500] = a[x][:2500]
    tok_b = np.concatenate([tok_a[:2500], rng.integers(0, 30000, 1500).astype(np.int32)])
    db = {x: b[x].cuda() for x in "qkvgb"}
    p, o, S = kda.prefill_cached(cache, pool, tok_b, *(db[x] for x in "qkvgb"), interval=1024)
    torch.cuda.synchronize()
    assert p == 2048                                       # resumed from A's checkpoint
    ro, rS, _ = oracle_run(b)
    assert o.shape[0] == 4000 - 2048
    assert rel(host(o), ro[2048:]) <= TOL and rel(host(S), rS) <= TOL

    # prompt A again: cached whole, nothing to run
    p, o, S = kda.prefill_cached(cache, pool, tok_a, *(da[x] for x in "qkvgb"), interval=1024)
    assert p == 3000 and o.shape[0] == 0
    ro, rS, _ = oracle_run(a)
    assert rel(host(S), rS) <= TOL
