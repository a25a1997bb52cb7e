"""The snapshot retention policy (kda_prefix_cache_*): longest-prefix lookup
over token ids, row reservation with eviction of interval checkpoints before
prompt-boundary ones (least recently used first), and the limits of a
reservation.  Host-side code of libkda; no GPU."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def kda():
    from linear_attention_serving_delta_gb300 import build, kda as binding
    build.build()
    binding.lib()
    return binding


def toks(n, seed):
    return np.random.default_rng(seed).integers(0, 50000, n).astype(np.int32)


def test_lookup_longest_prefix(kda):
    c = kda.PrefixCache(8)
    a = toks(300, 1)
    assert c.lookup(a) == (0, -1)
    rows = c.reserve(a, [64, 128, 300], [False, False, True])
    assert sorted(rows.tolist()) == [5, 6, 7] or len(set(rows.tolist())) == 3
    assert c.entries() == 3
    assert c.lookup(a) == (300, rows[2])
    assert c.lookup(a[:200]) == (128, rows[1])       # a prefix of the prompt
    assert c.lookup(a[:127]) == (64, rows[0])
    assert c.lookup(a[:63]) == (0, -1)
    b = a.copy()
    b[100] += 1                                       # diverges at token 100
    assert c.lookup(b) == (64, rows[0])
    b2 = np.concatenate([a, toks(50, 2)])             # extends the prompt
    assert c.lookup(b2) == (300, rows[2])
    assert c.lookup(np.zeros(0, np.int32)) == (0, -1)


def test_already_cached_positions_are_not_rewritten(kda):
    c = kda.PrefixCache(4)
    a = toks(256, 3)
    r1 = c.reserve(a, [64, 128], [False, False])
    assert (r1 >= 0).all()
    r2 = c.reserve(np.concatenate([a, toks(64, 4)]), [64, 128, 192], [False, False, True])
    assert r2[0] == -1 and r2[1] == -1 and r2[2] >= 0   # the first two are kept already
    assert c.entries() == 3


def test_eviction_prefers_interval_then_lru(kda):
    c = kda.PrefixCache(3)
    p1, p2, p3 = toks(128, 5), toks(128, 6), toks(128, 7)
    (r_end1,) = c.reserve(p1, [128], [True])              # boundary
    (r_mid2,) = c.reserve(p2, [64], [False])               # interval
    (r_mid3,) = c.reserve(p3, [64], [False])               # interval
    c.lookup(p2)                                           # p2's checkpoint becomes recent
    (r_new,) = c.reserve(toks(128, 8), [100], [True])
    assert r_new == r_mid3                                 # the LRU interval entry went first
    assert c.lookup(p3) == (0, -1)
    assert c.lookup(p1) == (128, r_end1)
    (r_new2,) = c.reserve(toks(128, 9), [90], [True])
    assert r_new2 == r_mid2                                # then the other interval entry
    (r_new3,) = c.reserve(toks(128, 10), [80], [True])
    assert r_new3 == r_new                                 # then the LRU boundary entry (p1's
    assert c.lookup(p1) == (128, r_end1)                   # was used by the lookup above)
    assert c.entries() == 3


def test_reservation_order_and_limits(kda):
    c = kda.PrefixCache(3)
    a = toks(512, 11)
    pos = [64, 128, 192, 256, 320, 512]
    rows = c.reserve(a, pos, [False] * 5 + [True])
    # three rows: the boundary first, then the latest interval positions
    assert rows[5] >= 0 and rows[4] >= 0 and rows[3] >= 0
    assert (rows[:3] == -1).all()
    assert c.lookup(a) == (512, rows[5])
    # keep_row: the row being resumed from is not evicted
    b = np.concatenate([a, toks(128, 12)])
    p, row = c.lookup(b)
    assert p == 512
    r = c.reserve(b, [576, 640], [False, True], keep_row=row)
    assert row not in r.tolist() and (r >= 0).all()
    assert c.lookup(a) == (512, row)


def test_invalid_arguments(kda):
    with pytest.raises(ValueError):
        kda.PrefixCache(0)
    c = kda.PrefixCache(2)
    a = toks(100, 13)
    for bad in ([0], [101], [50, 50], [60, 40]):
        with pytest.raises(ValueError):
            c.reserve(a, bad)
    with pytest.raises(ValueError):
        c.reserve(a, [10], keep_row=2)
    L = kda.lib()
    assert L.kda_prefix_cache_entries(None) == -1


def test_forget_frees_rows_of_a_failed_prefill(kda):
    """A reservation indexes its entries at once; if the prefill that was to
    write them fails, forget() drops them so no lookup resumes from an
    unwritten row, and the rows go back to the free list."""
    c = kda.PrefixCache(4)
    a = toks(256, 11)
    ok = c.reserve(a[:128], [64, 128], [False, True])
    assert c.lookup(a) == (128, ok[1])
    failed = c.reserve(a, [192, 256], [False, True])
    assert (failed >= 0).all() and c.entries() == 4
    assert c.lookup(a) == (256, failed[1])
    assert c.forget(np.concatenate([failed, [-1]])) == 2   # -1 entries are ignored
    assert c.entries() == 2
    assert c.lookup(a) == (128, ok[1])                       # back to the written prefix
    assert c.forget(failed) == 0                             # nothing left to drop
    # the freed rows are reused before any kept entry is evicted
    again = c.reserve(toks(200, 12), [100, 200], [False, True])
    assert sorted(again.tolist()) == sorted(failed.tolist())
    assert c.lookup(a) == (128, ok[1])
    with pytest.raises(ValueError):
        c.forget([4])                                        # outside the pool
    with pytest.raises(ValueError):
        c.forget([-2])


def test_prefill_cached_forgets_rows_when_the_call_fails(kda):
    """prefill_cached reserves rows before it builds and launches the prefill;
    when that raises (here: host tensors, refused by the binding before any
    launch), the reservation is dropped again, so the cache holds no entry
    for states that were never written."""
    import torch
    c = kda.PrefixCache(8)
    T, H, d = 300, 2, 16
    x = torch.zeros(T, H, d)
    pool = torch.zeros(8, H, d, d)
    with pytest.raises(ValueError):
        kda.prefill_cached(c, pool, toks(T, 21), x, x, x, x, torch.zeros(T, H), interval=128)
    assert c.entries() == 0
    assert c.lookup(toks(T, 21)) == (0, -1)
